// The PLE n-gram row-id hash on sm_103a: the head-lane kernel, for the tuned
// shapes whose heads divide a warp evenly (ngram_size 5 with 8 heads per
// order: 32 heads, one token a step; ngram_size 3 with 4: 8 heads, four
// tokens a step).
//
// The fixed-shape kernel (ple_rowids_fixed.cu) keeps one token per lane all
// the way through, so every lane reloads each head's constants from shared
// memory, and the rows go through a staged tile to reach coalesced stores.
// When a token's heads divide the warp's 32 lanes the hash can turn the warp
// around instead:
//   - the tile's windows are built one token per lane (the shared tile_windows
//     of ple_rowids_common.cuh), and each lane folds its token's mixes, one per
//     n-gram order, and stages them in shared memory (FreeToken PR #338,
//     "perf(ple): fuse the n-gram row-id hash into one Triton kernel", section
//     "What": the per-n-gram multiply / XOR loop);
//   - then lane l takes head l mod H for every (32 / H)-th token of the tile:
//     its head's remainder constants stay in its registers for the whole
//     layer, it reads its order's mix for each of its tokens (the lanes of one
//     order and token read one word: a broadcast), and the warp stores the
//     32 row ids of a step's tokens as one contiguous run of [L, T, H]
//     (256 bytes of int64, 128 of int32) -- the floored remainder plus
//     offset of section "What" / "Why it is safe".
// No block barrier, no shared constants, no staged readout: the warps of a
// block are independent from the start.  Every warp derives its own heads'
// reciprocals (four times the fixed-shape kernel's divisions), which the
// stores hide.  Measured on GB300 against the fixed-shape kernel, the
// 48-layer mixed batch: 17.25 -> 15.62 us in one launch, 16.41 -> 15.19 us
// reading an index, 16.84 -> 15.34 us with prepared constants (one-layer
// groups; two- and three-layer groups were slower).  The fully unrolled pass
// over a full tile keeps every offset a constant; int32 row ids gain from it
// (13.05 -> 12.58 us on the same batch), against a loss with a counted loop.
#include "ple_rowids_common.cuh"

namespace ple {
namespace {

constexpr int kHeadlaneTile = 32;

// Shared memory per warp: the staged ids (kHaloSlots + kTileTokens int64, the
// layout tile_windows expects) and the mixes, one row of N 8-byte words per
// token (N - 1 orders and a pad word: an odd row pitch, so the lanes' 8-byte
// stores of one order hit distinct banks, and the four words one token's
// orders occupy are read without conflict).
__host__ __device__ constexpr size_t headlane_warp_bytes(int N) {
    return (size_t)(kHaloSlots + kTileTokens) * 8 + (size_t)kHeadlaneTile * N * 8;
}

// A row id stored with the streaming hint: int64, or its low 32 bits.
template <typename OutT>
__device__ __forceinline__ void st_row(OutT* p, int64_t v) {
    if constexpr (sizeof(OutT) == 8)
        __stcs(reinterpret_cast<long long*>(p), (long long)v);
    else
        __stcs(reinterpret_cast<int*>(p), (int)v);
}

template <typename IdT, int NT, int HPT, bool kCarry, int kIdx, typename OutT>
__global__ void __launch_bounds__(kMaxWarps * 32, kFixedMinBlocks)
row_ids_headlane_kernel(const RowIdsParams p) {
    constexpr int N = NT;
    constexpr int H = (NT - 1) * HPT;
    static_assert(32 % H == 0, "the heads divide the warp");
    constexpr int TPS = 32 / H;  // tokens per hash step
    const int G = p.group_layers;
    const int l0 = blockIdx.y * G;
    const int gl = min(G, p.L - l0);
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    extern __shared__ __align__(16) unsigned char smem[];
    wait_prior_grid();
    if constexpr (kCarry) carry_empty_requests<IdT>(p, N);
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kHeadlaneTile;
    const int ntile = (int)max((int64_t)0, min((int64_t)kHeadlaneTile, p.T - t0));
    if (ntile == 0) return;  // no block barrier follows
    unsigned char* wbase = smem + (size_t)warp * headlane_warp_bytes(N);
    int64_t* ids_s = reinterpret_cast<int64_t*>(wbase) + kHaloSlots;
    uint2* mix_s = reinterpret_cast<uint2*>(wbase + (size_t)(kHaloSlots + kTileTokens) * 8);
    int64_t VA[N], VB[N];
    tile_windows<IdT, N, kHeadlaneTile, kIdx, kCarry>(p, ids_s, t0, ntile, lane, VA, VB);

    const int head = lane % H;
    const int sub = lane / H;         // which of the step's tokens
    const int order = head / HPT;     // head h is of order n = order + 2
#pragma unroll 1
    for (int l = 0; l < gl; ++l) {
        const int64_t layer = (int64_t)l0 + l;
        // this lane's head's constants, loaded (prepared) or derived, while
        // the lane folds its token's mixes
        const int64_t k = layer * H + head;
        const HeadConst c = p.heads != nullptr ? load_head_const(p.heads, k)
                                               : make_head_const(p.vocab[k], p.offsets[k]);
        const long long* ml = reinterpret_cast<const long long*>(p.mult) + layer * N;
        uint64_t mix = (uint64_t)VA[0] * (uint64_t)__ldg(ml);
#pragma unroll
        for (int s = 1; s < N; ++s) {
            // order n = s + 1 folds shifts 0..s; staged in offset binary
            mix ^= (uint64_t)VA[s] * (uint64_t)__ldg(ml + s);
            const OffsetBinary u = offset_binary(mix);
            mix_s[lane * N + (s - 1)] = make_uint2(u.lo, u.hi);
        }
        __syncwarp();
        OutT* dst = static_cast<OutT*>(p.out) + (layer * p.T + t0 + sub) * H + head;
        const uint2* mrow = mix_s + sub * N + order;
        if (c.ext.z == kHeadFast) {
            const uint32_t nv = (uint32_t)((int32_t)c.fast.z >> 1);  // -v
            if (ntile == kHeadlaneTile) {
                // a full tile: every step's offsets are compile-time
#pragma unroll
                for (int i = 0; i < kHeadlaneTile / TPS; ++i) {
                    const uint2 w = mrow[i * TPS * N];
                    st_row<OutT>(dst + i * TPS * H,
                           (int64_t)((uint64_t)c.off +
                                       floormod_fast(OffsetBinary{w.x, w.y}, c.fast, nv)));
                }
            } else {
#pragma unroll 1
                for (int i = 0; sub + i * TPS < ntile; ++i) {
                    const uint2 w = mrow[i * TPS * N];
                    st_row<OutT>(dst + i * TPS * H,
                           (int64_t)((uint64_t)c.off +
                                       floormod_fast(OffsetBinary{w.x, w.y}, c.fast, nv)));
                }
            }
        } else {
#pragma unroll 1
            for (int i = 0; sub + i * TPS < ntile; ++i) {
                const uint2 w = mrow[i * TPS * N];
                st_row<OutT>(dst + i * TPS * H,
                       (int64_t)row_general(OffsetBinary{w.x, w.y}, c.fast, c.off, c.ext));
            }
        }
        __syncwarp();  // the next layer overwrites the staged mixes
    }
}

template <typename IdT, int NT, int HPT, bool kCarry, typename OutT>
KernelFn pick_headlane(int mode) {
    if (mode == kIdxDecode) return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxDecode, OutT>;
    if (mode == kIdxCu) return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxCu, OutT>;
    return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxArrays, OutT>;
}

template <typename IdT, int NT, int HPT, typename OutT>
KernelFn pick_headlane(bool carry, int mode) {
    return carry ? pick_headlane<IdT, NT, HPT, true, OutT>(mode)
                 : pick_headlane<IdT, NT, HPT, false, OutT>(mode);
}

template <typename IdT>
KernelFn pick_headlane(int N, int out_bytes, bool carry, int mode) {
    if (out_bytes == 4) return pick_headlane<IdT, 5, 8, int32_t>(carry, mode);
    return N == 3 ? pick_headlane<IdT, 3, 4, int64_t>(carry, mode)
                  : pick_headlane<IdT, 5, 8, int64_t>(carry, mode);
}

}  // namespace

// The tuned shapes whose heads divide the warp evenly: 32 heads (one token a
// step), int64 or int32 row ids, and 8 heads (four tokens a step), int64 row
// ids.  Measured on GB300 against the fixed-shape kernel: the ragged
// 16-request batch (8 heads) 2.90 -> 2.43 us a call; the 48-layer mixed
// batch with int32 row ids 13.05 -> 12.58 us.  The 12-head shape stays on the
// fixed-shape kernel: with 32 row ids a pass each lane needs three heads'
// constants and the large prefill took 27.6 us with prepared constants
// against 22.1 (int32 row ids), 57.7 against 30.4 us with int64 ones and
// derived constants (every warp dividing for three heads a layer).
bool uses_headlane_kernel(const RowIdsParams& p) {
    return (p.N == 5 && p.hpn == 8) || (p.N == 3 && p.hpn == 4 && p.out_bytes == 8);
}

size_t headlane_smem_bytes(int N, int warps) { return (size_t)warps * headlane_warp_bytes(N); }

int headlane_tile_tokens() { return kHeadlaneTile; }

cudaError_t launch_row_ids_headlane(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                    cudaStream_t stream) {
    const bool carry = p.next_ctx != nullptr;
    const KernelFn fn = id_bytes == 4
                            ? pick_headlane<int32_t>(p.N, p.out_bytes, carry, p.index_mode)
                            : pick_headlane<int64_t>(p.N, p.out_bytes, carry, p.index_mode);
    return launch_fn(fn, p, cfg, stream);
}

}  // namespace ple
