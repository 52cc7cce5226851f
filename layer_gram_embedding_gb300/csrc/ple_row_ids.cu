// The PLE n-gram row-id hash kernel for sm_103a.
//
// Computes, for every token of a ragged batch and every layer, head and
// n-gram order, the table row id of FreeToken PR #338 ("perf(ple): fuse the
// n-gram row-id hash into one Triton kernel", section "What"):
//
//   V(t,s) = W(t,s) while no boundary id lies among W(t,1..s), else the
//            boundary id (first observation: the whole-window cummax scan
//            only ever looks ngram_size-1 places back, so the predicate is
//            carried over at most ngram_size-1 steps);
//   W(t,s) = ids[t-s] if local[t] >= s, else the carried context
//            ngram_context[req[t]][ctx_len + local[t] - s] (second
//            observation: the packed window is never built);
//   row    = floormod(XOR_{s<n} V(t,s)*M[l][s], vocab[l][h]) + off[l][h].
//
// Work decomposition (one GPU, HBM-bound: 8*L*H bytes of row ids are written
// per token against 16 bytes read):
//   - grid.x covers the tokens in warp tiles of 64 (two per lane); grid.y
//     splits the layers into groups so that even a small T fills the SMs.
//   - Block prologue: the group's per-head divisor constants (one reciprocal
//     per head, see ple_divmod.cuh) and multipliers go to shared memory.
//   - Each warp stages its tile's ids plus an ngram_size-1 halo in shared
//     memory (16-byte vector loads when aligned), then per 32-token half:
//     builds V in registers with the carried boundary predicate, and per
//     layer hashes every head into a shared staging tile whose odd row pitch
//     makes the per-token writes bank-conflict free, then streams the tile
//     out as contiguous, fully coalesced 8-byte stores ([L, T, H] layout:
//     one warp-half covers 32*H consecutive int64).
//   - No inter-warp communication after the prologue (warp-per-tile), no
//     atomics, no host reads: the launch is graph-capturable.
#include <stdint.h>

#include "ple.h"
#include "ple_divmod.cuh"
#include "ple_internal.h"

namespace ple {
namespace {

template <typename IdT>
__device__ __forceinline__ int64_t load_id(const IdT* p, int64_t i);

template <>
__device__ __forceinline__ int64_t load_id<int64_t>(const int64_t* p, int64_t i) {
    return (int64_t)__ldg(reinterpret_cast<const long long*>(p) + i);
}

template <>
__device__ __forceinline__ int64_t load_id<int32_t>(const int32_t* p, int64_t i) {
    return (int64_t)__ldg(p + i);
}

// A full 64-token tile of ids, 16-byte vector loads (tile base 16B-aligned).
template <typename IdT>
__device__ __forceinline__ void load_tile_vec(const IdT* src, int64_t* dst, int lane);

template <>
__device__ __forceinline__ void load_tile_vec<int64_t>(const int64_t* src, int64_t* dst, int lane) {
    // 64 ids = 512 bytes = one 16-byte load per lane
    const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(src) + lane);
    reinterpret_cast<longlong2*>(dst)[lane] = v;
}

template <>
__device__ __forceinline__ void load_tile_vec<int32_t>(const int32_t* src, int64_t* dst, int lane) {
    // 64 ids = 256 bytes = one 16-byte load for each of 16 lanes
    if (lane < 16) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(src) + lane);
        longlong2* d = reinterpret_cast<longlong2*>(dst) + 2 * lane;
        d[0] = make_longlong2((long long)v.x, (long long)v.y);
        d[1] = make_longlong2((long long)v.z, (long long)v.w);
    }
}

// Hash one layer for this lane's token into its staging row.
template <int NMAX, int NT, bool kFast>
__device__ __forceinline__ void hash_layer(const int64_t (&V)[NMAX], int N, int hpn,
                                           const int64_t* __restrict__ ml,
                                           const HeadConst* __restrict__ hl,
                                           int64_t* __restrict__ srow) {
    uint64_t mix = (uint64_t)V[0] * (uint64_t)ml[0];
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
        if (NT == 0 && s >= N) break;
        // order n = s + 1 folds shifts 0..s
        mix ^= (uint64_t)V[s] * (uint64_t)ml[s];
        const Magnitude x = magnitude((int64_t)mix);
        const HeadConst* hs = hl + (s - 1) * hpn;
        int64_t* so = srow + (s - 1) * hpn;
#pragma unroll 4
        for (int j = 0; j < hpn; ++j) {
            if (kFast) {
                const uint4 c = *reinterpret_cast<const uint4*>(hs + j);
                so[j] = row_fast_positive(x, c.x, c.y, c.z, hs[j].off);
            } else {
                so[j] = row_general(x, hs[j]);
            }
        }
    }
}

template <typename IdT, int NT>
__global__ void __launch_bounds__(kMaxWarps * 32)
row_ids_kernel(const RowIdsParams p) {
    constexpr int NMAX = NT > 0 ? NT : PLE_MAX_NGRAM;
    const int N = NT > 0 ? NT : p.N;
    const int H = p.H;
    const int hpn = p.hpn;
    const int pitch = p.stage_pitch;
    const int G = p.group_layers;
    const int l0 = blockIdx.y * G;
    const int gl = min(G, p.L - l0);
    const int nwarps = blockDim.x >> 5;

    extern __shared__ __align__(16) unsigned char smem[];
    HeadConst* hc = reinterpret_cast<HeadConst*>(smem);
    int64_t* mul_s = reinterpret_cast<int64_t*>(smem + (size_t)G * H * sizeof(HeadConst));
    int64_t* ids_all = mul_s + ((G * N + 1) & ~1);
    int64_t* stage_all = ids_all + nwarps * (kHaloSlots + kTileTokens);

    // ---- block prologue: this layer group's divisor constants and multipliers
    int fast = 1;
    for (int i = threadIdx.x; i < gl * H; i += blockDim.x) {
        const int64_t k = (int64_t)l0 * H + i;
        const HeadConst c = make_head_const(p.vocab[k], p.offsets[k]);
        hc[i] = c;
        fast &= (c.kind == kHeadFast) ? 1 : 0;
    }
    for (int i = threadIdx.x; i < gl * N; i += blockDim.x) mul_s[i] = p.mult[(int64_t)l0 * N + i];
    const bool all_fast = __syncthreads_and(fast) != 0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kTileTokens;
    if (t0 >= p.T) return;
    const int ntile = (int)min((int64_t)kTileTokens, p.T - t0);
    int64_t* ids_s = ids_all + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
    int64_t* stage = stage_all + (size_t)warp * 32 * pitch;
    const IdT* ids = static_cast<const IdT*>(p.ids);
    const IdT* ctx = static_cast<const IdT*>(p.ctx);
    const int64_t b = p.boundary;

    // ---- stage the tile's ids and the N-1 ids left of it
    if (ntile == kTileTokens && p.ids_vec_ok) {
        load_tile_vec<IdT>(ids + t0, ids_s, lane);
    } else {
        for (int i = lane; i < ntile; i += 32) ids_s[i] = load_id<IdT>(ids, t0 + i);
    }
    if (lane < N - 1 && t0 - 1 - lane >= 0) ids_s[-1 - lane] = load_id<IdT>(ids, t0 - 1 - lane);
    __syncwarp();

    // staging readout walk: element e of a 32*H run sits at row e / H, column e % H
    const int dq = 32 / H;
    const int dr = 32 % H;
    const int q0 = lane / H;
    const int r0 = lane % H;

#pragma unroll 1
    for (int u = 0; u < kTileTokens / 32; ++u) {
        const int nsub = min(32, ntile - 32 * u);
        if (nsub <= 0) break;
        const int i = 32 * u + lane;
        const int64_t t = t0 + i;
        const bool live = lane < nsub;

        // ---- the window and the carried boundary predicate
        int64_t V[NMAX];
        {
            int32_t r = 0, q = 0;
            if (live) {
                r = __ldg(p.req + t);
                q = __ldg(p.local + t);
            }
            // keep device-side index data inside the ranges that can be addressed
            r = min(max(r, 0), p.B - 1);
            q = (int32_t)min((int64_t)max(q, 0), t);
            V[0] = live ? ids_s[i] : 0;
            const IdT* crow = ctx + (int64_t)r * (N - 1) + (N - 1) + q;
            bool valid = true;
#pragma unroll
            for (int s = 1; s < NMAX; ++s) {
                if (NT == 0 && s >= N) break;
                const int64_t w = (q >= s) ? ids_s[i - s] : load_id<IdT>(crow, -s);
                valid = valid && (w != b);
                V[s] = valid ? w : b;
            }
        }

        // ---- every layer of the group: hash into staging, stream out
#pragma unroll 1
        for (int l = 0; l < gl; ++l) {
            if (all_fast)
                hash_layer<NMAX, NT, true>(V, N, hpn, mul_s + l * N, hc + l * H, stage + lane * pitch);
            else
                hash_layer<NMAX, NT, false>(V, N, hpn, mul_s + l * N, hc + l * H, stage + lane * pitch);
            __syncwarp();
            long long* dst = reinterpret_cast<long long*>(p.out) +
                             ((int64_t)(l0 + l) * p.T + t0 + 32 * u) * H;
            const int nel = nsub * H;
            int qq = q0, rr = r0;
            for (int e = lane; e < nel; e += 32) {
                __stcs(dst + e, (long long)stage[qq * pitch + rr]);
                rr += dr;
                qq += dq;
                if (rr >= H) {
                    rr -= H;
                    ++qq;
                }
            }
            __syncwarp();
        }
    }
}

template <typename IdT>
using KernelFn = void (*)(const RowIdsParams);

template <typename IdT>
KernelFn<IdT> pick_kernel(int N) {
    switch (N) {
        case 2: return row_ids_kernel<IdT, 2>;
        case 3: return row_ids_kernel<IdT, 3>;
        case 4: return row_ids_kernel<IdT, 4>;
        case 5: return row_ids_kernel<IdT, 5>;
        case 6: return row_ids_kernel<IdT, 6>;
        case 7: return row_ids_kernel<IdT, 7>;
        case 8: return row_ids_kernel<IdT, 8>;
        default: return row_ids_kernel<IdT, 0>;
    }
}

template <typename IdT>
cudaError_t launch_typed(const RowIdsParams& p, const RowIdsLaunch& cfg, cudaStream_t stream) {
    const KernelFn<IdT> fn = pick_kernel<IdT>(p.N);
    if (cfg.smem_bytes > 48 * 1024) {
        // Opting in to more than 48 KB of dynamic shared memory is a function
        // attribute; setting it is idempotent and not a stream operation.
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    fn<<<cfg.grid, cfg.block, cfg.smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

RowIdsLaunch plan_row_ids(RowIdsParams& p, const DeviceFacts& dev) {
    RowIdsLaunch cfg;
    const int64_t tiles = (p.T + kTileTokens - 1) / kTileTokens;
    int warps = (int)(tiles < kMaxWarps ? tiles : kMaxWarps);
    p.stage_pitch = p.H | 1;
    const size_t per_warp = (size_t)(kHaloSlots + kTileTokens) * 8 + (size_t)32 * p.stage_pitch * 8;

    // layer groups: split the layers until there are ~8 blocks per SM, so the
    // last wave is short even when T alone gives few tiles; constants stay
    // within their shared-memory budget
    int64_t blocks_x = (tiles + warps - 1) / warps;
    const int64_t target = 8 * (int64_t)dev.sm_count;
    int64_t groups = (target + blocks_x - 1) / blocks_x;
    if (groups < 1) groups = 1;
    if (groups > p.L) groups = p.L;
    int G = (int)((p.L + groups - 1) / groups);
    const int g_cap = (int)(kConstBudgetBytes / ((size_t)p.H * sizeof(HeadConst)));
    if (G > g_cap) G = g_cap > 0 ? g_cap : 1;
    groups = (p.L + G - 1) / G;
    p.group_layers = G;

    const size_t fixed = (size_t)G * p.H * sizeof(HeadConst) + round_up((size_t)G * p.N, 2) * 8;
    while (warps > 1 && fixed + warps * per_warp > (size_t)dev.max_smem_optin) --warps;
    blocks_x = (tiles + warps - 1) / warps;
    cfg.grid = dim3((unsigned)blocks_x, (unsigned)groups, 1);
    cfg.block = dim3(32 * warps, 1, 1);
    cfg.smem_bytes = fixed + warps * per_warp;
    return cfg;
}

cudaError_t launch_row_ids(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                           cudaStream_t stream) {
    if (id_bytes == 4) return launch_typed<int32_t>(p, cfg, stream);
    return launch_typed<int64_t>(p, cfg, stream);
}

}  // namespace ple
