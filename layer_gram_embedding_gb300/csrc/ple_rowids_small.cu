// The PLE n-gram row-id hash on sm_103a: the small-batch kernel.
//
// Decode steps and short prefills are latency-bound: a call's time is the
// launch plus the longest chain of dependent steps inside it, not bytes.
// The tiled kernels (ple_rowids_fixed.cu, ple_rowids_runtime.cu) spend that
// chain on a block prologue -- each head's reciprocal, shared-memory staging
// of ids and constants, a block barrier, a staged readout -- which pays off
// only when a block then hashes thousands of row ids.  This kernel gives each
// row id (token t, layer l, head h) its own thread instead:
//   - block (heads_per_ngram, ngram_size - 1, tokens): threadIdx.x is the head
//     j within its order, threadIdx.y the order n - 2, threadIdx.z the token,
//     so h = (n - 2) * heads_per_ngram + j needs no division; grid.y is the
//     layer.  Consecutive threads own consecutive row ids of [L, T, H].
//   - the thread reads its window W(t, 0..n-1) straight from global memory
//     (FreeToken PR #338, "perf(ple): fuse the n-gram row-id hash into one
//     Triton kernel", section "What", second observation: ids[t-s] while
//     local[t] >= s, else the carried context row), carries the boundary
//     predicate over the shifts (first observation), and loads its head's
//     prepared constants (ple_prepare_heads) or computes the reciprocal
//     itself, in parallel with the window loads;
//   - no shared memory, no barrier, one store per thread.
// The arithmetic is the tiled kernels': the same window rule, the same
// Barrett remainder (ple_divmod.cuh), so the row ids are identical.
#include "ple_rowids_common.cuh"

namespace ple {
namespace {

// kIdx and kPrepared are compile-time: as run-time branches, the index
// choice alone added about 0.15 us to a decode call (measured on GB300).
template <typename IdT, int NT, int kIdx, bool kPrepared>
__global__ void __launch_bounds__(kSmallMaxThreads)
row_ids_small_kernel(const RowIdsParams p) {
    constexpr int NMAX = NT > 0 ? NT : PLE_MAX_NGRAM;
    const int N = NT > 0 ? NT : p.N;
    wait_prior_grid();
    carry_empty_requests<IdT>(p, N);
    const int64_t t = (int64_t)blockIdx.x * blockDim.z + threadIdx.z;
    if (t >= p.T) return;
    const int l = blockIdx.y;
    const int o = threadIdx.y;  // order n = o + 2 folds shifts 0..o+1
    const int h = o * p.hpn + threadIdx.x;
    const int64_t k = (int64_t)l * p.H + h;
    // prepared constants are three loads; otherwise the head's reciprocal is
    // computed here, in parallel with the window loads
    const int64_t vocab = kPrepared ? 0 : __ldg(reinterpret_cast<const long long*>(p.vocab) + k);
    const int64_t off = kPrepared ? 0 : __ldg(reinterpret_cast<const long long*>(p.offsets) + k);

    int32_t r, q;
    load_index<kIdx>(p, t, true, r, q);
    const IdT* ids = static_cast<const IdT*>(p.ids);
    const IdT* crow = static_cast<const IdT*>(p.ctx) + (int64_t)r * (N - 1) + (N - 1) + q;
    const long long* ml = reinterpret_cast<const long long*>(p.mult) + (int64_t)l * N;
    int64_t w[NMAX];
    w[0] = load_id<IdT>(ids, t);
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
        if (NT == 0 && s >= N) break;
        // q is clamped to [0, t], so t - s >= 0 on the first branch and the
        // context index stays inside row r on the second
        w[s] = s <= o + 1 ? (q >= s ? load_id<IdT>(ids, t - s) : load_id<IdT>(crow, -s)) : 0;
    }
    const HeadConst c = kPrepared ? load_head_const(p.heads, k) : make_head_const(vocab, off);

    uint64_t mix = (uint64_t)w[0] * (uint64_t)__ldg(ml);
    bool valid = true;
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
        if ((NT == 0 && s >= N) || s > o + 1) break;
        valid = valid && (w[s] != p.boundary);
        mix ^= (uint64_t)(valid ? w[s] : p.boundary) * (uint64_t)__ldg(ml + s);
    }
    const OffsetBinary u = offset_binary(mix);
    const int64_t row = (c.ext.z & kHeadFast) ? row_fast(u, c.fast, c.off)
                                              : row_general(u, c.fast, c.off, c.ext);
    const int64_t e = ((int64_t)l * p.T + t) * p.H + h;
    if (p.out_bytes == 8)
        __stcs(static_cast<long long*>(p.out) + e, (long long)row);
    else
        __stcs(static_cast<int*>(p.out) + e, (int)row);

    // the context carry, once per token: the request's last token writes the
    // last N-1 ids of (context row, its tokens), oldest first
    if (p.next_ctx != nullptr && l == 0 && h == 0) {
        if (p.cu != nullptr && t != (int64_t)__ldg(p.cu + r + 1) - 1) return;
        IdT* dst = static_cast<IdT*>(p.next_ctx) + (int64_t)r * (N - 1);
        for (int cc = 0; cc < N - 1; ++cc) {
            const int s = N - 2 - cc;
            dst[cc] = (q >= s) ? ids[t - s] : crow[-s];
        }
    }
}

template <typename IdT, int kIdx, bool kPrepared>
KernelFn pick_small(int N) {
    switch (N) {
        case 3: return row_ids_small_kernel<IdT, 3, kIdx, kPrepared>;
        case 4: return row_ids_small_kernel<IdT, 4, kIdx, kPrepared>;
        case 5: return row_ids_small_kernel<IdT, 5, kIdx, kPrepared>;
        default: return row_ids_small_kernel<IdT, 0, kIdx, kPrepared>;
    }
}

template <typename IdT, int kIdx>
KernelFn pick_small(const RowIdsParams& p) {
    return p.heads != nullptr ? pick_small<IdT, kIdx, true>(p.N)
                              : pick_small<IdT, kIdx, false>(p.N);
}

template <typename IdT>
KernelFn pick_small(const RowIdsParams& p) {
    if (p.index_mode == kIdxDecode) return pick_small<IdT, kIdxDecode>(p);
    if (p.index_mode == kIdxCu) return pick_small<IdT, kIdxCu>(p);
    return pick_small<IdT, kIdxArrays>(p);
}

}  // namespace

bool small_batch_fits(const RowIdsParams& p) {
    // T * H * L <= kSmallMaxRows without overflow (T < 2^31, H <= 256)
    const int64_t per_layer = p.T * p.H;
    return per_layer > 0 && per_layer <= kSmallMaxRows && p.L <= kSmallMaxRows / per_layer &&
           p.L <= 65535;
}

RowIdsLaunch plan_small(RowIdsParams& p) {
    RowIdsLaunch cfg;
    int tpb = kSmallBlockThreads / p.H;
    tpb = tpb < 1 ? 1 : tpb > 64 ? 64 : tpb;  // blockDim.z is at most 64
    cfg.grid = dim3((unsigned)((p.T + tpb - 1) / tpb), (unsigned)p.L, 1);
    cfg.block = dim3((unsigned)p.hpn, (unsigned)(p.N - 1), (unsigned)tpb);
    cfg.smem_bytes = 0;
    cfg.small = true;
    p.group_layers = 1;
    p.stage_pitch = p.H | 1;
    return cfg;
}

cudaError_t launch_row_ids_small(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                 cudaStream_t stream) {
    const KernelFn fn = id_bytes == 4 ? pick_small<int32_t>(p) : pick_small<int64_t>(p);
    return launch_fn(fn, p, cfg, stream);
}

}  // namespace ple
