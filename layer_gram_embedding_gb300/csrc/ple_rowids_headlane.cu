// The PLE n-gram row-id hash on sm_103a: the head-lane kernel, for the tuned
// shapes whose row ids a warp can store 32 at a time in global order.
//
// The fixed-shape kernel (ple_rowids_fixed.cu) keeps one token per lane all
// the way through, so every lane reloads each head's constants from shared
// memory, and the rows go through a staged tile to reach coalesced stores.
// The head-lane kernel turns the warp around instead:
//   - the tile's windows are built one token per lane (the shared tile_windows
//     of ple_rowids_common.cuh), and each lane folds its token's mixes, one per
//     n-gram order, and stages them in shared memory (FreeToken PR #338,
//     "perf(ple): fuse the n-gram row-id hash into one Triton kernel", section
//     "What": the per-n-gram multiply / XOR loop);
//   - then the warp writes the tile's [32 tokens, H heads] block of row ids
//     in passes of 32 consecutive ones: in pass k lane l hashes row 32k + l,
//     head (32k + l) mod H of token (32k + l) / H, reading that token's mix
//     for the head's order (a broadcast among the lanes that share it), and
//     the pass is one contiguous store (256 bytes of int64 row ids, 128 of
//     int32) -- the floored remainder plus offset of section "What" / "Why it
//     is safe".  A lane meets H / gcd(32, H) distinct heads: one when the
//     heads divide the warp (32 or 8 heads), three for 12 heads.
// Over a full tile the passes are unrolled, so every mix and store offset is a
// constant.  The heads' remainder constants come one of two ways:
//   - per warp (one head a lane): each lane derives or loads its head's
//     constants itself and keeps them in registers for the layer; no block
//     barrier at all;
//   - per block (kShared): as in the fixed-shape kernel, the block's threads
//     derive each head's constants once into shared memory behind one
//     barrier, and each lane reads its heads' from there every layer.
// Measured on GB300 against the fixed-shape kernel (interleaved A/B, µs per
// call): the 48-layer mixed batch, per warp, 17.25 -> 15.62 in one launch,
// 16.41 -> 15.19 reading an index, 16.84 -> 15.34 with prepared constants, and
// its int32 variant, per block, 12.66 -> 11.00 (10.60 with its two plain adds
// as ALU add-mins, floormod_fast_alu); the ragged batch (8 heads, per
// warp) 2.90 -> 2.43; the large prefill (12 heads, per block) 30.43 -> 29.92.
// The other combinations stay on the fixed-shape kernel (they measured slower
// here): the large prefill's int32 variant (23.5 against 22.3) and the 8-head
// shape's int32 rows.
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
    return (size_t)(kHaloSlots + kTileTokens) * 8 + (size_t)kHeadlaneTile * (N | 1) * 8;
}

__host__ __device__ constexpr int gcd_c(int a, int b) { return b == 0 ? a : gcd_c(b, a % b); }



// A row id stored with the streaming hint: int64, or its low 32 bits.
template <typename OutT>
__device__ __forceinline__ void st_row(OutT* p, int64_t v) {
    if constexpr (sizeof(OutT) == 8)
        __stcs(reinterpret_cast<long long*>(p), (long long)v);
    else
        __stcs(reinterpret_cast<int*>(p), (int)v);
}

// One lane's token: fold its mixes for every order of one layer and stage
// them in offset binary (order n = s + 1 folds shifts 0..s), order s - 1 at
// mix_s[row + (s - 1) * OS].
template <int N, int OS = 1, typename MulT>
__device__ __forceinline__ void stage_mixes(const int64_t (&V)[N], MulT ml, uint2* mix_s, int row) {
    uint64_t mix = (uint64_t)V[0] * (uint64_t)ml(0);
#pragma unroll
    for (int s = 1; s < N; ++s) {
        mix ^= (uint64_t)V[s] * (uint64_t)ml(s);
        const OffsetBinary u = offset_binary(mix);
        mix_s[row + (s - 1) * OS] = make_uint2(u.lo, u.hi);
    }
}

// The layers with per-warp constants (one head a lane: H divides 32): lane l
// hashes head l mod H of tokens l / H, l / H + 32 / H, ...
template <int N, int H, int HPT, typename OutT>
__device__ __forceinline__ void hash_layers_own(const RowIdsParams& p, uint2* mix_s,
                                                const int64_t (&VA)[N], int l0, int gl,
                                                int64_t t0, int ntile, int lane, OutT* out) {
    constexpr int TPS = 32 / H;  // tokens a pass
    constexpr int P = N | 1;
    const int head = lane % H;
    const int sub = lane / H;
    const int order = head / HPT;  // head h is of order n = order + 2
#pragma unroll 1
    for (int l = 0; l < gl; ++l) {
        const int64_t layer = (int64_t)l0 + l;
        // this lane's head's constants, loaded (prepared) or derived, while
        // the lane folds its token's mixes
        const int64_t k = layer * H + head;
        const HeadConst c = p.heads != nullptr ? load_head_const(p.heads, k)
                                               : make_head_const(p.vocab[k], p.offsets[k]);
        const long long* ml = reinterpret_cast<const long long*>(p.mult) + layer * N;
        stage_mixes<N>(VA, [&](int s) { return (int64_t)__ldg(ml + s); }, mix_s, lane * P);
        __syncwarp();
        OutT* dst = out + (layer * p.T + t0 + sub) * H + head;
        const uint2* mrow = mix_s + sub * P + order;
        if (c.ext.z == kHeadFast) {
            const uint32_t nv = (uint32_t)((int32_t)c.fast.z >> 1);  // -v
            if (ntile == kHeadlaneTile) {
                // a full tile: every pass's offsets are compile-time
#pragma unroll
                for (int i = 0; i < kHeadlaneTile / TPS; ++i) {
                    const uint2 w = mrow[i * TPS * P];
                    st_row(dst + i * TPS * H,
                           (int64_t)((uint64_t)c.off +
                                     floormod_fast_alu(OffsetBinary{w.x, w.y}, c.fast, nv,
                                                       p.ones)));
                }
            } else {
#pragma unroll 1
                for (int i = 0; sub + i * TPS < ntile; ++i) {
                    const uint2 w = mrow[i * TPS * P];
                    st_row(dst + i * TPS * H,
                           (int64_t)((uint64_t)c.off +
                                     floormod_fast(OffsetBinary{w.x, w.y}, c.fast, nv)));
                }
            }
        } else {
#pragma unroll 1
            for (int i = 0; sub + i * TPS < ntile; ++i) {
                const uint2 w = mrow[i * TPS * P];
                st_row(dst + i * TPS * H, row_general(OffsetBinary{w.x, w.y}, c.fast, c.off, c.ext));
            }
        }
        __syncwarp();  // the next layer overwrites the staged mixes
    }
}

// The layers with the block's constants in shared memory: pass k covers row
// ids 32k .. 32k + 31 of the tile's [32, H] block, lane l's being row 32k + l,
// head (32k + l) mod H, token (32k + l) / H -- for k = j + NH q, head j's
// (32j + l) mod H and token (32j + l) / H + ADV q (head, mbase per j).
template <int N, int H, int HPT, int NH, int ADV, int P, typename OutT>
__device__ __forceinline__ void hash_layers_shared(const RowIdsParams& p, const SmemLayout& sm,
                                                   uint2* mix_s, const int64_t (&VA)[N], int l0,
                                                   int gl, int64_t t0, int ntile, int lane,
                                                   bool all_fast, const int (&head)[NH],
                                                   const int (&mbase)[NH], OutT* out) {
#pragma unroll 1
    for (int l = 0; l < gl; ++l) {
        const int64_t layer = (int64_t)l0 + l;
        const int64_t* ml = sm.mul + l * N;
        // at 32 heads a lane hashes one head, so one order, of every token:
        // the mixes are staged order-major (pitch 34 words, 16-byte aligned
        // rows whose starts fall 4 banks apart) and a 16-byte load brings two
        // consecutive tokens' mixes
        constexpr bool kOM = H == 32;
        constexpr int PO = kHeadlaneTile + 2;
        static_assert(!kOM || (N - 2) * PO + kHeadlaneTile <= kHeadlaneTile * P,
                      "order-major mixes stay within the warp's staging rows");
        if constexpr (kOM)
            stage_mixes<N, PO>(VA, [&](int s) { return ml[s]; }, mix_s, lane);
        else
            stage_mixes<N>(VA, [&](int s) { return ml[s]; }, mix_s, lane * P);
        __syncwarp();
        OutT* dst = out + (layer * p.T + t0) * H + lane;
        if (all_fast && ntile == kHeadlaneTile) {
            uint4 cf[NH];
            int64_t coff[NH];
            uint32_t nv[NH];
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                cf[j] = sm.fast[l * H + head[j]];
                coff[j] = sm.off[l * H + head[j]];
                nv[j] = (uint32_t)((int32_t)cf[j].z >> 1);  // -v
            }
            // the sign-fix add, and for int32 rows the offset add too, as
            // add-mins on the ALU (floormod_fast_alu)
            if constexpr (kOM) {
                const uint4* mq = reinterpret_cast<const uint4*>(mix_s + (lane / HPT) * PO);
#pragma unroll
                for (int i = 0; i < kHeadlaneTile / 2; ++i) {
                    const uint4 w = mq[i];  // tokens 2i and 2i + 1
                    const uint32_t r0 =
                        floormod_fast_alu(OffsetBinary{w.x, w.y}, cf[0], nv[0], p.ones);
                    const uint32_t r1 =
                        floormod_fast_alu(OffsetBinary{w.z, w.w}, cf[0], nv[0], p.ones);
                    if constexpr (sizeof(OutT) == 4) {
                        st_row(dst + 64 * i, (int64_t)min((uint32_t)coff[0] + r0, p.ones));
                        st_row(dst + 64 * i + 32, (int64_t)min((uint32_t)coff[0] + r1, p.ones));
                    } else {
                        st_row(dst + 64 * i, (int64_t)((uint64_t)coff[0] + r0));
                        st_row(dst + 64 * i + 32, (int64_t)((uint64_t)coff[0] + r1));
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < H; ++k) {
                    const int j = k % NH, q = k / NH;
                    const uint2 w = mix_s[mbase[j] + ADV * q * P];
                    const uint32_t r =
                        floormod_fast_alu(OffsetBinary{w.x, w.y}, cf[j], nv[j], p.ones);
                    if constexpr (sizeof(OutT) == 4)
                        st_row(dst + 32 * k, (int64_t)min((uint32_t)coff[j] + r, p.ones));
                    else
                        st_row(dst + 32 * k, (int64_t)((uint64_t)coff[j] + r));
                }
            }
        } else {
            // a partial tile, or a head of the group off the 32-bit fast path
#pragma unroll 1
            for (int k = 0; k < H; ++k) {
                const int r = 32 * (k % NH) + lane;
                const int t = r / H + ADV * (k / NH);
                if (t < ntile) {
                    const int i = l * H + r % H;
                    const uint2 w = kOM ? mix_s[((r % H) / HPT) * PO + t]
                                        : mix_s[t * P + (r % H) / HPT];
                    const OffsetBinary u{w.x, w.y};
                    st_row(dst + 32 * k, sm.ext[i].z == kHeadFast
                                             ? row_fast(u, sm.fast[i], sm.off[i])
                                             : row_general(u, sm.fast[i], sm.off[i], sm.ext[i]));
                }
            }
        }
        __syncwarp();  // the next layer overwrites the staged mixes
    }
}

template <typename IdT, int NT, int HPT, bool kCarry, int kIdx, typename OutT, bool kShared>
__global__ void __launch_bounds__(kMaxWarps * 32, kFixedMinBlocks)
row_ids_headlane_kernel(const RowIdsParams p) {
    constexpr int N = NT;
    constexpr int H = (NT - 1) * HPT;
    static_assert(H <= 32, "at most one head per lane");
    constexpr int GG = gcd_c(32, H);
    constexpr int NH = H / GG;    // distinct heads a lane hashes
    constexpr int ADV = 32 / GG;  // tokens its passes advance every NH passes
    constexpr int P = N | 1;      // staged mix row pitch (odd)
    static_assert(kShared || NH == 1, "per-warp constants hold one head a lane");
    const int G = p.group_layers;
    const int l0 = blockIdx.y * G;
    const int gl = min(G, p.L - l0);
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    extern __shared__ __align__(16) unsigned char smem[];
    wait_prior_grid();
    if constexpr (kCarry) carry_empty_requests<IdT>(p, N);
    SmemLayout sm{};
    int fast_vote = 1;
    if constexpr (kShared) {
        sm = carve_smem(smem, G, H, N, nwarps);
        fast_vote = load_group_constants(p, sm, l0, gl, H, N);
    }
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kHeadlaneTile;
    const int ntile = (int)max((int64_t)0, min((int64_t)kHeadlaneTile, p.T - t0));
    int64_t* ids_s;
    uint2* mix_s;
    if constexpr (kShared) {
        ids_s = sm.ids + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
        mix_s = reinterpret_cast<uint2*>(sm.stage + (size_t)warp * kHeadlaneTile * P * 8);
    } else {
        unsigned char* wbase = smem + (size_t)warp * headlane_warp_bytes(N);
        ids_s = reinterpret_cast<int64_t*>(wbase) + kHaloSlots;
        mix_s = reinterpret_cast<uint2*>(wbase + (size_t)(kHaloSlots + kTileTokens) * 8);
    }
    int64_t VA[N], VB[N];
    bool all_fast = true;
    if constexpr (kShared) {
        // the block's constants are published once its windows' loads are in
        // flight, so the divisions overlap them
        if (ntile > 0)
            tile_windows<IdT, N, kHeadlaneTile, kIdx, kCarry>(p, ids_s, t0, ntile, lane, VA, VB);
        all_fast = __syncthreads_and(fast_vote) != 0;
        if (ntile == 0) return;
    } else {
        if (ntile == 0) return;  // no block barrier follows
        tile_windows<IdT, N, kHeadlaneTile, kIdx, kCarry>(p, ids_s, t0, ntile, lane, VA, VB);
    }

    if constexpr (kShared) {
        // head j of this lane's passes, and where its token's mix row starts
        int head[NH], mbase[NH];
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            head[j] = (32 * j + lane) % H;
            mbase[j] = ((32 * j + lane) / H) * P + head[j] / HPT;  // order n = head / hpn + 2
        }
        hash_layers_shared<N, H, HPT, NH, ADV, P>(p, sm, mix_s, VA, l0, gl, t0, ntile, lane,
                                                   all_fast, head, mbase,
                                                   static_cast<OutT*>(p.out));
    } else {
        hash_layers_own<N, H, HPT>(p, mix_s, VA, l0, gl, t0, ntile, lane,
                                   static_cast<OutT*>(p.out));
    }
}

template <typename IdT, int NT, int HPT, bool kCarry, typename OutT, bool kShared>
KernelFn pick_headlane(int mode) {
    if (mode == kIdxDecode)
        return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxDecode, OutT, kShared>;
    if (mode == kIdxCu) return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxCu, OutT, kShared>;
    return row_ids_headlane_kernel<IdT, NT, HPT, kCarry, kIdxArrays, OutT, kShared>;
}

template <typename IdT, int NT, int HPT, typename OutT, bool kShared>
KernelFn pick_headlane(bool carry, int mode) {
    return carry ? pick_headlane<IdT, NT, HPT, true, OutT, kShared>(mode)
                 : pick_headlane<IdT, NT, HPT, false, OutT, kShared>(mode);
}

// (5,8) int64 per warp, (5,8) int32 per block, (3,4) int64 per warp,
// (4,4) int64 per block -- the choices uses_headlane_kernel and
// headlane_shared_constants make.
template <typename IdT>
KernelFn pick_headlane(int N, int out_bytes, bool carry, int mode) {
    if (N == 5)
        return out_bytes == 4 ? pick_headlane<IdT, 5, 8, int32_t, true>(carry, mode)
                              : pick_headlane<IdT, 5, 8, int64_t, false>(carry, mode);
    if (N == 3) return pick_headlane<IdT, 3, 4, int64_t, false>(carry, mode);
    return pick_headlane<IdT, 4, 4, int64_t, true>(carry, mode);
}

}  // namespace

// The shapes whose heads divide the warp evenly among the tuned ones, with
// int64 row ids: 32 heads (one token a step) and 8 (four).  Measured on
// GB300 against the fixed-shape kernel: the ragged 16-request batch (8 heads)
// 2.90 -> 2.43 us a call.  With int32 row ids the fixed-shape kernel
// measured faster (the 48-layer mixed batch 13.1 us against 13.7-14.7 us
// here at any layer grouping: every warp derives its own heads' reciprocals,
// and half-size stores do not hide that), and so did the 12-head shape,
// where a step's 24 lanes leave 8 idle and its 192-byte stores straddle
// cache lines (the large prefill 29.9 -> 41.9 us).
bool uses_headlane_kernel(const RowIdsParams& p) {
    if (p.N == 5 && p.hpn == 8) return true;
    return p.out_bytes == 8 && ((p.N == 3 && p.hpn == 4) || (p.N == 4 && p.hpn == 4));
}

bool headlane_shared_constants(const RowIdsParams& p) { return p.N == 4 || p.out_bytes == 4; }

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
