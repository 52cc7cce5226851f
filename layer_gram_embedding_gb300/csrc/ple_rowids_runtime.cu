// The PLE n-gram row-id hash on sm_103a: the runtime-shape kernel, the launch
// plan and the dispatch between it, the fixed-shape kernel and the
// small-batch kernel (ple_rowids_small.cu).
//
// The runtime-shape kernel serves every (ngram_size, heads_per_ngram) the
// fixed-shape kernel is not compiled for, and the index-free decode: one
// token per lane per 32-token half tile, int64 rows staged in shared memory
// with an odd row pitch (H | 1, conflict-free 8-byte stores), read out in
// global order with 8-byte stores.  The window, the carried boundary
// predicate, the per-head Barrett remainder and the context carry are the
// shared code of ple_rowids_common.cuh.
#include "ple_rowids_common.cuh"

namespace ple {
namespace {

// Any shape: one token per lane per half tile, int64 staging with odd pitch.
template <typename IdT, int NT, typename OutT>
__global__ void __launch_bounds__(kMaxWarps * 32)
row_ids_kernel(const RowIdsParams p) {
    constexpr int NMAX = NT > 0 ? NT : PLE_MAX_NGRAM;
    const int N = NT > 0 ? NT : p.N;
    const int H = p.H;
    const int hpn = p.hpn;
    const int pitch = H | 1;
    const int G = p.group_layers;
    const int l0 = blockIdx.y * G;
    const int gl = min(G, p.L - l0);
    const int nwarps = blockDim.x >> 5;

    extern __shared__ __align__(16) unsigned char smem[];
    wait_prior_grid();
    carry_empty_requests<IdT>(p, N);
    const SmemLayout sm = carve_smem(smem, G, H, N, nwarps);
    const int fast_vote = load_group_constants(p, sm, l0, gl, H, N);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kTileTokens;
    const int ntile = (int)max((int64_t)0, min((int64_t)kTileTokens, p.T - t0));
    int64_t* ids_s = sm.ids + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
    int64_t* stage = reinterpret_cast<int64_t*>(sm.stage + (size_t)warp * stage_bytes(H, false));
    const bool carry = p.next_ctx != nullptr && blockIdx.y == 0;
    if (ntile > 0) stage_ids<IdT>(p, ids_s, t0, ntile, N, lane);
    const bool all_fast = __syncthreads_and(fast_vote) != 0;
    if (ntile == 0) return;

#pragma unroll 1
    for (int u = 0; u < kTileTokens / 32; ++u) {
        const int nsub = min(32, ntile - 32 * u);
        if (nsub <= 0) break;
        int64_t V[NMAX];
        int32_t r, q;
        if (p.index_mode == kIdxDecode)
            window<IdT, NMAX, NT, kIdxDecode>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, V, r,
                                              q);
        else if (p.index_mode == kIdxCu)
            window<IdT, NMAX, NT, kIdxCu>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, V, r, q);
        else
            window<IdT, NMAX, NT, kIdxArrays>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, V, r,
                                              q);
        if (carry) carry_context<IdT>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, r, q);
#pragma unroll 1
        for (int l = 0; l < gl; ++l) {
            const int hb = l * H;
            if (all_fast)
                hash_layer<NMAX, NT, true>(V, N, hpn, sm.mul + l * N, sm.fast + hb, sm.off + hb,
                                           sm.ext + hb, stage + lane * pitch);
            else
                hash_layer<NMAX, NT, false>(V, N, hpn, sm.mul + l * N, sm.fast + hb, sm.off + hb,
                                            sm.ext + hb, stage + lane * pitch);
            __syncwarp();
            OutT* dst = static_cast<OutT*>(p.out) + ((int64_t)(l0 + l) * p.T + t0 + 32 * u) * H;
            readout_runtime<OutT>(stage, dst, lane, nsub, H, pitch);
            __syncwarp();
        }
    }
}

// The runtime-shape kernel for ngram_size N (N > 8 runs the generic loop).
template <typename IdT, typename OutT>
KernelFn pick_runtime_kernel(int N) {
    switch (N) {
        case 2: return row_ids_kernel<IdT, 2, OutT>;
        case 3: return row_ids_kernel<IdT, 3, OutT>;
        case 4: return row_ids_kernel<IdT, 4, OutT>;
        case 5: return row_ids_kernel<IdT, 5, OutT>;
        case 6: return row_ids_kernel<IdT, 6, OutT>;
        case 7: return row_ids_kernel<IdT, 7, OutT>;
        case 8: return row_ids_kernel<IdT, 8, OutT>;
        default: return row_ids_kernel<IdT, 0, OutT>;
    }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

bool shape_is_fixed(int N, int hpn) {
    return (N == 3 && (hpn == 2 || hpn == 4)) || (N == 4 && hpn == 4) || (N == 5 && hpn == 8);
}

// The fixed-shape kernel takes the tuned shapes, the runtime-shape kernel
// every other one.
static bool uses_fixed_kernel(const RowIdsParams& p) { return shape_is_fixed(p.N, p.hpn); }

RowIdsLaunch plan_row_ids(RowIdsParams& p, const DeviceFacts& dev, bool runtime_layout) {
    if (!runtime_layout && small_batch_fits(p)) return plan_small(p);
    RowIdsLaunch cfg;
    cfg.small = false;
    const bool fixed_shape = !runtime_layout && uses_fixed_kernel(p);
    const bool headlane = fixed_shape && uses_headlane_kernel(p);
    const int tile = headlane      ? headlane_tile_tokens()
                     : fixed_shape ? fixed_tile_tokens(p.H)
                                   : kTileTokens;
    const int64_t tiles = (p.T + tile - 1) / tile;
    int warps = (int)(tiles < kMaxWarps ? tiles : kMaxWarps);
    p.stage_pitch = p.H | 1;
    const size_t per_warp = headlane ? headlane_smem_bytes(p.N, 1)
                                     : (size_t)(kHaloSlots + kTileTokens) * 8 +
                                           stage_bytes(p.H, fixed_shape);

    // layer groups: split the layers until there are per_sm blocks per SM,
    // so the last wave is short even when T alone gives few tiles; constants
    // stay within their shared-memory budget
    int64_t blocks_x = (tiles + warps - 1) / warps;
    const int per_sm = runtime_layout       ? kTargetBlocksPerSmEmbed
                       : p.out_bytes == 8 ? kTargetBlocksPerSmI64
                                          : kTargetBlocksPerSm;
    const int64_t target = per_sm * (int64_t)dev.sm_count;
    int64_t groups = (target + blocks_x - 1) / blocks_x;
    if (groups < 1) groups = 1;
    if (groups > p.L) groups = p.L;
    int G = (int)((p.L + groups - 1) / groups);
    const int g_cap = (int)(kConstBudgetBytes / head_const_bytes(p.H));
    if (G > g_cap) G = g_cap > 0 ? g_cap : 1;
    groups = (p.L + G - 1) / G;
    p.group_layers = G;

    // a head-lane kernel with per-warp constants keeps them in registers
    const size_t fixed = headlane && !headlane_shared_constants(p)
                             ? 0
                             : head_const_bytes(G * p.H) + round_up((size_t)G * p.N, 2) * 8;
    while (warps > 1 && fixed + warps * per_warp > (size_t)dev.max_smem_optin) --warps;
    // a small grid (a medium batch with few layers) spreads its warp tiles
    // over more SMs with fewer warps per block
    while (warps > 1 && ((tiles + warps - 1) / warps) * groups <
                            (int64_t)kSpreadBlocksPerSm * dev.sm_count)
        --warps;
    blocks_x = (tiles + warps - 1) / warps;
    cfg.grid = dim3((unsigned)blocks_x, (unsigned)groups, 1);
    cfg.block = dim3(32 * warps, 1, 1);
    cfg.smem_bytes = fixed + warps * per_warp;
    return cfg;
}

cudaError_t launch_row_ids(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                           cudaStream_t stream) {
    if (cfg.small) return launch_row_ids_small(p, id_bytes, cfg, stream);
    if (uses_fixed_kernel(p) && uses_headlane_kernel(p))
        return launch_row_ids_headlane(p, id_bytes, cfg, stream);
    if (uses_fixed_kernel(p)) return launch_row_ids_fixed(p, id_bytes, cfg, stream);
    KernelFn fn;
    if (p.out_bytes == 4)
        fn = id_bytes == 4 ? pick_runtime_kernel<int32_t, int32_t>(p.N)
                           : pick_runtime_kernel<int64_t, int32_t>(p.N);
    else
        fn = id_bytes == 4 ? pick_runtime_kernel<int32_t, int64_t>(p.N)
                           : pick_runtime_kernel<int64_t, int64_t>(p.N);
    return launch_fn(fn, p, cfg, stream);
}

}  // namespace ple
