// The PLE n-gram row-id hash on sm_103a: the fixed-shape kernel.
//
// Compiled for the PLE configurations this library is tuned for -- (ngram
// size, heads per order) in {(3,2), (3,4), (4,4), (5,8)}, each with int32 or
// int64 ids, int64 or int32 row ids, with or without the context carry, and
// each way of finding a token's request (an index, a decode without one, a
// search of cu_seqlens) -- every choice at compile time, because a run-time
// branch in the window costs the large prefill.
// Each lane hashes two tokens of the 64-token tile (lane and lane + 32) per
// shared constant load; the fast path stages 32-bit remainders as head pairs
// in rows of odd pitch (8-byte stores hit 16 distinct bank pairs per half
// warp) -- or, for int32 row ids, as swizzled head quads (16-byte stores and
// loads without bank conflicts) -- and the readout walks the tile in global
// order ([L, T, H]), adds each head's offset in registers and stores 16 bytes
// per lane, so a warp store covers 512 consecutive bytes.  Shapes with more
// than 16 heads stage one 32-token half (a 16-token quarter on the general
// path) at a time, and in the cu_seqlens search mode take 32-token tiles.
// Heads off the 32-bit fast path (vocab outside (0, 2^29]) stage int64 rows
// and read them out 8 bytes at a time.  The (5,8) shape, and (3,4) and (4,4)
// with int64 row ids, run the head-lane kernel instead
// (ple_rowids_headlane.cu).
#include "ple_rowids_common.cuh"

namespace ple {
namespace {

__host__ __device__ constexpr int gcd_const(int a, int b) { return b == 0 ? a : gcd_const(b, a % b); }

// Fixed shapes with an even number of heads per order (the PLE
// configurations this library is tuned for).  Each lane hashes two tokens of
// the 64-token tile (lane and lane + 32) per constant load; the fast path
// stages 32-bit remainders as pairs of heads, and the readout adds the head
// offsets in registers and stores 16 bytes per lane in global order.
template <int K, int P2, int NC, int GSTEP, bool kVec, bool kFull>
__device__ __forceinline__ void readout_pairs(const uint2* __restrict__ st,
                                              long long* __restrict__ dst, int lane, int nsub,
                                              const int (&soff)[K], const int (&stok)[K],
                                              const longlong2 (&offs)[NC]) {
    longlong2* d2 = reinterpret_cast<longlong2*>(dst);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        if (kFull || stok[j] < nsub) {
            const uint2 r = st[soff[j]];
            const longlong2 o = offs[((32 * j) % K) / GSTEP];
            const longlong2 rows = make_longlong2((long long)((unsigned long long)o.x + r.x),
                                                  (long long)((unsigned long long)o.y + r.y));
            if (kVec) {
                __stcs(d2 + 32 * j + lane, rows);
            } else {
                long long* d1 = reinterpret_cast<long long*>(d2 + 32 * j + lane);
                __stcs(d1, rows.x);
                __stcs(d1 + 1, rows.y);
            }
        }
    }
}

// int32 row ids of the split staging (more than 16 heads, pair staging):
// four heads (two staged pairs) per 16-byte lane store; the offsets' low
// words are added in 32-bit arithmetic (the low 32 bits of the int64 row
// id).  K2 quads per token.  At 32 heads the pitch of 17 pairs puts the two
// tokens a half warp reads in opposite bank parities, so the pair loads are
// conflict-free.
template <int K2, int P2, int NC, int GSTEP, bool kVec, bool kFull>
__device__ __forceinline__ void readout_quads(const uint2* __restrict__ st, int* __restrict__ dst,
                                              int lane, int nsub, const int (&soff)[K2],
                                              const int (&stok)[K2], const int4 (&offs)[NC]) {
    int4* d4 = reinterpret_cast<int4*>(dst);
#pragma unroll
    for (int j = 0; j < K2; ++j) {
        if (kFull || stok[j] < nsub) {
            const uint2 a = st[soff[j]];
            const uint2 b = st[soff[j] + 1];
            const int4 o = offs[((32 * j) % K2) / GSTEP];
            const int4 rows = make_int4((int)((unsigned)o.x + a.x), (int)((unsigned)o.y + a.y),
                                        (int)((unsigned)o.z + b.x), (int)((unsigned)o.w + b.y));
            if (kVec) {
                __stcs(d4 + 32 * j + lane, rows);
            } else {
                int* d1 = reinterpret_cast<int*>(d4 + 32 * j + lane);
                __stcs(d1, rows.x);
                __stcs(d1 + 1, rows.y);
                __stcs(d1 + 2, rows.z);
                __stcs(d1 + 3, rows.w);
            }
        }
    }
}

// Quad staging of int32 remainders (shapes of at most 16 heads): four heads
// per 16-byte slot, K2 = H / 4 slots per token, no padding, slot index
// token * K2 + (quad ^ quad_swizzle(token)).  A 16-byte shared access is
// served eight lanes at a time, conflict-free when the eight slots differ
// modulo 8: for odd K2 consecutive tokens already do, both when a lane
// stores its own token's quads and when the readout's lanes walk the tile
// in global order; for K2 a power of two the quad index is XORed with the
// token's rank among the 8 / K2 tokens one readout phase covers.  The
// swizzle repeats every 32 tokens, so the tile's second half uses the same.
template <int K2>
__device__ __forceinline__ int quad_swizzle(int token) {
    static_assert(K2 % 2 == 1 || K2 == 2 || K2 == 4 || K2 == 8, "quad staging layout");
    if constexpr (K2 % 2 == 1)
        return 0;
    else
        return (token / (8 / K2)) % K2;
}

// int32 row ids from quad staging: one 16-byte shared load per 16-byte
// global store (K2 per lane per half tile).
template <int K2, int NC, int GSTEP, bool kVec, bool kFull>
__device__ __forceinline__ void readout_quad_slots(const uint4* __restrict__ st,
                                                   int* __restrict__ dst, int lane, int nsub,
                                                   const int (&soff)[K2], const int (&stok)[K2],
                                                   const int4 (&offs)[NC]) {
    int4* d4 = reinterpret_cast<int4*>(dst);
#pragma unroll
    for (int j = 0; j < K2; ++j) {
        if (kFull || stok[j] < nsub) {
            const uint4 a = st[soff[j]];
            const int4 o = offs[((32 * j) % K2) / GSTEP];
            const int4 rows = make_int4((int)((unsigned)o.x + a.x), (int)((unsigned)o.y + a.y),
                                        (int)((unsigned)o.z + a.z), (int)((unsigned)o.w + a.w));
            if (kVec) {
                __stcs(d4 + 32 * j + lane, rows);
            } else {
                int* d1 = reinterpret_cast<int*>(d4 + 32 * j + lane);
                __stcs(d1, rows.x);
                __stcs(d1 + 1, rows.y);
                __stcs(d1 + 2, rows.z);
                __stcs(d1 + 3, rows.w);
            }
        }
    }
}

// One staged half tile (32 rows) of the split staging, read out for the
// output type: the head offsets of this lane's columns, then 16-byte stores.
template <typename OutT, int KU, int P2, int NU, int GU>
__device__ __forceinline__ void split_readout(const uint2* __restrict__ st, OutT* dst, int lane,
                                              int nsub, bool vec_out, const int (&soff)[KU],
                                              const int (&stok)[KU], const SmemLayout& sm,
                                              int hb, int r0) {
    if constexpr (sizeof(OutT) == 8) {
        longlong2 offs[NU];
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            int col = r0 + k * GU;
            col = col >= KU ? col - KU : col;
            offs[k] = *reinterpret_cast<const longlong2*>(sm.off + hb + 2 * col);
        }
        long long* d = reinterpret_cast<long long*>(dst);
        if (vec_out && nsub == 32)
            readout_pairs<KU, P2, NU, GU, true, true>(st, d, lane, 32, soff, stok, offs);
        else if (vec_out)
            readout_pairs<KU, P2, NU, GU, true, false>(st, d, lane, nsub, soff, stok, offs);
        else
            readout_pairs<KU, P2, NU, GU, false, false>(st, d, lane, nsub, soff, stok, offs);
    } else {
        int4 offs[NU];
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            int col = r0 + k * GU;
            col = col >= KU ? col - KU : col;
            offs[k] = *reinterpret_cast<const int4*>(sm.off32 + hb + 4 * col);
        }
        int* d = reinterpret_cast<int*>(dst);
        if (vec_out && nsub == 32)
            readout_quads<KU, P2, NU, GU, true, true>(st, d, lane, 32, soff, stok, offs);
        else if (vec_out)
            readout_quads<KU, P2, NU, GU, true, false>(st, d, lane, nsub, soff, stok, offs);
        else
            readout_quads<KU, P2, NU, GU, false, false>(st, d, lane, nsub, soff, stok, offs);
    }
}

template <typename IdT, int NT, int HPT, typename OutT, bool kCarry, int kIdx>
__global__ void __launch_bounds__(kMaxWarps * 32, kFixedMinBlocks)
row_ids_fixed_kernel(const RowIdsParams p) {
    static_assert(NT >= 2 && HPT >= 2 && HPT % 2 == 0, "fixed shapes have even heads_per_ngram");
    constexpr int N = NT;
    constexpr int H = (NT - 1) * HPT;
    constexpr int K = H / 2;        // 16-byte output chunks (head pairs) per token
    constexpr int P2 = K | 1;       // staging row pitch in 8-byte pairs (odd)
    constexpr int PG = H | 1;       // int64 staging pitch for the general path (odd)
    static_assert(K <= 32, "readout walk assumes K <= 32");
    const int G = p.group_layers;
    const int l0 = blockIdx.y * G;
    const int gl = min(G, p.L - l0);
    const int nwarps = blockDim.x >> 5;

    extern __shared__ __align__(16) unsigned char smem[];
    wait_prior_grid();
    if constexpr (kCarry) carry_empty_requests<IdT>(p, N);
    const SmemLayout sm = carve_smem(smem, G, H, N, nwarps);
    const int fast_vote = load_group_constants(p, sm, l0, gl, H, N);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kTile = fixed_tile_tokens(H);  // 64, or 32 (see there)
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kTile;
    const int ntile = (int)max((int64_t)0, min((int64_t)kTile, p.T - t0));
    int64_t* ids_s = sm.ids + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
    unsigned char* stage = sm.stage + (size_t)warp * stage_bytes(H, true);
    const int nA = min(32, ntile);
    const int nB = ntile - 32;  // tokens in the second half (may be <= 0)
    int64_t VA[N], VB[N];
    if (ntile > 0) tile_windows<IdT, N, kTile, kIdx, kCarry>(p, ids_s, t0, ntile, lane, VA, VB);
    const bool all_fast = __syncthreads_and(fast_vote) != 0;
    if (ntile == 0) return;

    if (!all_fast) {
        // some head of this group is off the fast path: int64 rows, 8-byte
        // readout, RG tokens at a time (a half tile, or a quarter when the
        // staging is split)
        constexpr int RG = general_stage_rows(H);
        int64_t* st = reinterpret_cast<int64_t*>(stage);
#pragma unroll 1
        for (int u = 0; u < 2; ++u) {
            const int nsub = u == 0 ? nA : nB;
#pragma unroll 1
            for (int q0 = 0; q0 < 32; q0 += RG) {
                const int nq = min(RG, nsub - q0);
                if (nq <= 0) break;
                const bool mine = RG == 32 || (lane >= q0 && lane < q0 + RG);
#pragma unroll 1
                for (int l = 0; l < gl; ++l) {
                    const int hb = l * H;
                    if (mine)
                        hash_layer<N, N, false>(u == 0 ? VA : VB, N, HPT, sm.mul + l * N,
                                                sm.fast + hb, sm.off + hb, sm.ext + hb,
                                                st + (lane - q0) * PG);
                    __syncwarp();
                    OutT* dst = static_cast<OutT*>(p.out) +
                                ((int64_t)(l0 + l) * p.T + t0 + 32 * u + q0) * H;
                    readout_runtime<OutT>(st, dst, lane, nq, H, PG);
                    __syncwarp();
                }
            }
        }
        return;
    }

    const uint2* stA = reinterpret_cast<const uint2*>(stage);
    uint2* stAw = reinterpret_cast<uint2*>(stage);
    // readout walk, the same for every layer: a 16-byte store carries U staged
    // pairs (1 for int64, 2 for int32), KU such units per token; unit c =
    // 32 j + lane of a half tile is token c / KU, column c % KU; with
    // q0 = lane / KU, r0 = lane % KU the step j adds the compile-time
    // (32 j) / KU and (32 j) % KU, carrying one token when the column wraps
    constexpr int U = sizeof(OutT) == 8 ? 1 : 2;
    static_assert(K % U == 0, "int32 output needs a multiple of 4 heads");
    constexpr int KU = K / U;
    constexpr int GU = gcd_const(32, KU);
    constexpr int NU = KU / GU;
    const int q0 = lane / KU;
    const int r0 = lane % KU;
    // int32 row ids of shapes without split staging stage quads (see
    // quad_swizzle); soff then counts 16-byte slots, else 8-byte pairs
    constexpr bool kQuadStage = U == 2 && fast_stage_rows(H) == 64;
    int soff[KU], stok[KU];
#pragma unroll
    for (int j = 0; j < KU; ++j) {
        const int cj = (32 * j) % KU;
        // cj == 0 (KU divides 32) folds the carry away: the offsets are then
        // affine in j and need no registers of their own
        const bool carry = cj != 0 && r0 + cj >= KU;
        const int col = r0 + cj - (carry ? KU : 0);
        stok[j] = q0 + (32 * j) / KU + (carry ? 1 : 0);
        if constexpr (kQuadStage)
            soff[j] = stok[j] * KU + (col ^ quad_swizzle<KU>(stok[j]));
        else
            soff[j] = stok[j] * P2 + U * col;
    }
    const bool full = nA == 32 && nB == 32;
    const bool vec_out = p.out_vec_ok != 0;

    if constexpr (fast_stage_rows(H) == 32) {
        // split staging: hash and read out one half tile at a time
#pragma unroll 1
        for (int l = 0; l < gl; ++l) {
            const int64_t* ml = sm.mul + l * N;
            const uint4* hf = sm.fast + l * H;
            OutT* dst = static_cast<OutT*>(p.out) + ((int64_t)(l0 + l) * p.T + t0) * H;
#pragma unroll 1
            for (int u = 0; u < 2; ++u) {
                const int nsub = u == 0 ? nA : nB;
                if (nsub <= 0) break;
                // select element by element: the windows stay in registers
                uint64_t mix = (uint64_t)(u == 0 ? VA[0] : VB[0]) * (uint64_t)ml[0];
#pragma unroll
                for (int s = 1; s < N; ++s) {
                    mix ^= (uint64_t)(u == 0 ? VA[s] : VB[s]) * (uint64_t)ml[s];
                    const OffsetBinary uu = offset_binary(mix);
#pragma unroll
                    for (int j = 0; j < HPT; j += 2) {
                        const int h = (s - 1) * HPT + j;
                        const uint4 c0 = hf[h];
                        const uint4 c1 = hf[h + 1];
                        stAw[lane * P2 + h / 2] = make_uint2(
                            floormod_fast(uu, c0, (uint32_t)((int32_t)c0.z >> 1)),
                            floormod_fast(uu, c1, (uint32_t)((int32_t)c1.z >> 1)));
                    }
                }
                __syncwarp();
                split_readout<OutT, KU, P2, NU, GU>(stA, dst + 32 * u * H, lane, nsub, vec_out,
                                                    soff, stok, sm, l * H, r0);
                __syncwarp();
            }
        }
    } else if constexpr (kQuadStage) {
        // int32 row ids: each lane stages its two tokens' remainders four
        // heads to a 16-byte store, and the readout takes one 16-byte load
        // per 16-byte global store (with pair staging, the readout's pair
        // loads met 3-way bank conflicts at 12 heads and made the shared
        // memory pipe the bound)
        uint4* stQ = reinterpret_cast<uint4*>(stage);
        const int sw = quad_swizzle<KU>(lane);  // token 32 + lane's too
#pragma unroll 1
        for (int l = 0; l < gl; ++l) {
            const int64_t* ml = sm.mul + l * N;
            const uint4* hf = sm.fast + l * H;
            uint64_t mixA = (uint64_t)VA[0] * (uint64_t)ml[0];
            uint64_t mixB = (uint64_t)VB[0] * (uint64_t)ml[0];
            uint32_t rA[H], rB[H];
#pragma unroll
            for (int s = 1; s < N; ++s) {
                const uint64_t m = (uint64_t)ml[s];
                mixA ^= (uint64_t)VA[s] * m;
                mixB ^= (uint64_t)VB[s] * m;
                const OffsetBinary uA = offset_binary(mixA);
                const OffsetBinary uB = offset_binary(mixB);
#pragma unroll
                for (int j = 0; j < HPT; j += 2) {
                    const int h = (s - 1) * HPT + j;
                    const uint4 c0 = hf[h];
                    const uint4 c1 = hf[h + 1];
                    const uint32_t n0 = (uint32_t)((int32_t)c0.z >> 1);  // -v of each head
                    const uint32_t n1 = (uint32_t)((int32_t)c1.z >> 1);
                    rA[h] = floormod_fast_alu(uA, c0, n0, p.ones);
                    rA[h + 1] = floormod_fast_alu(uA, c1, n1, p.ones);
                    rB[h] = floormod_fast_alu(uB, c0, n0, p.ones);
                    rB[h + 1] = floormod_fast_alu(uB, c1, n1, p.ones);
                    if (h % 4 == 2) {
                        // heads h - 2 .. h + 1 complete quad h / 4
                        const int qd = (h / 4) ^ sw;
                        stQ[lane * KU + qd] = make_uint4(rA[h - 2], rA[h - 1], rA[h], rA[h + 1]);
                        stQ[(32 + lane) * KU + qd] =
                            make_uint4(rB[h - 2], rB[h - 1], rB[h], rB[h + 1]);
                    }
                }
            }
            __syncwarp();
            int4 offs[NU];
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                int col = r0 + k * GU;
                col = col >= KU ? col - KU : col;
                offs[k] = *reinterpret_cast<const int4*>(sm.off32 + l * H + 4 * col);
            }
            int* d = reinterpret_cast<int*>(static_cast<OutT*>(p.out) +
                                            ((int64_t)(l0 + l) * p.T + t0) * H);
            if (full && vec_out) {
                readout_quad_slots<KU, NU, GU, true, true>(stQ, d, lane, 32, soff, stok, offs);
                readout_quad_slots<KU, NU, GU, true, true>(stQ + 32 * KU, d + 32 * H, lane, 32,
                                                           soff, stok, offs);
            } else if (vec_out) {
                readout_quad_slots<KU, NU, GU, true, false>(stQ, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_quad_slots<KU, NU, GU, true, false>(stQ + 32 * KU, d + 32 * H, lane,
                                                                nB, soff, stok, offs);
            } else {
                readout_quad_slots<KU, NU, GU, false, false>(stQ, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_quad_slots<KU, NU, GU, false, false>(stQ + 32 * KU, d + 32 * H, lane,
                                                                 nB, soff, stok, offs);
            }
            __syncwarp();
        }
    } else {
        // int64 row ids: pair staging, 16-byte readout of one pair per store
#pragma unroll 1
        for (int l = 0; l < gl; ++l) {
            const int64_t* ml = sm.mul + l * N;
            const uint4* hf = sm.fast + l * H;
            uint64_t mixA = (uint64_t)VA[0] * (uint64_t)ml[0];
            uint64_t mixB = (uint64_t)VB[0] * (uint64_t)ml[0];
#pragma unroll
            for (int s = 1; s < N; ++s) {
                const uint64_t m = (uint64_t)ml[s];
                mixA ^= (uint64_t)VA[s] * m;
                mixB ^= (uint64_t)VB[s] * m;
                const OffsetBinary uA = offset_binary(mixA);
                const OffsetBinary uB = offset_binary(mixB);
#pragma unroll
                for (int j = 0; j < HPT; j += 2) {
                    const int h = (s - 1) * HPT + j;
                    const uint4 c0 = hf[h];
                    const uint4 c1 = hf[h + 1];
                    const uint32_t n0 = (uint32_t)((int32_t)c0.z >> 1);  // -v of each head
                    const uint32_t n1 = (uint32_t)((int32_t)c1.z >> 1);
                    stAw[lane * P2 + h / 2] =
                        make_uint2(floormod_fast(uA, c0, n0), floormod_fast(uA, c1, n1));
                    stAw[(32 + lane) * P2 + h / 2] =
                        make_uint2(floormod_fast(uB, c0, n0), floormod_fast(uB, c1, n1));
                }
            }
            __syncwarp();
            OutT* dst = static_cast<OutT*>(p.out) + ((int64_t)(l0 + l) * p.T + t0) * H;
            // this lane's readout columns' offsets for layer l
            longlong2 offs[NU];
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                int col = r0 + k * GU;
                col = col >= KU ? col - KU : col;
                offs[k] = *reinterpret_cast<const longlong2*>(sm.off + l * H + 2 * col);
            }
            long long* d = reinterpret_cast<long long*>(dst);
            if (full && vec_out) {
                readout_pairs<KU, P2, NU, GU, true, true>(stA, d, lane, 32, soff, stok, offs);
                readout_pairs<KU, P2, NU, GU, true, true>(stA + 32 * P2, d + 32 * H, lane, 32,
                                                         soff, stok, offs);
            } else if (vec_out) {
                readout_pairs<KU, P2, NU, GU, true, false>(stA, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_pairs<KU, P2, NU, GU, true, false>(stA + 32 * P2, d + 32 * H, lane,
                                                              nB, soff, stok, offs);
            } else {
                readout_pairs<KU, P2, NU, GU, false, false>(stA, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_pairs<KU, P2, NU, GU, false, false>(stA + 32 * P2, d + 32 * H, lane,
                                                               nB, soff, stok, offs);
            }
            __syncwarp();
        }
    }
}

template <typename IdT, typename OutT, bool kCarry, int kIdx>
KernelFn pick_fixed(int N, int hpn) {
    if (N == 3 && hpn == 2) return row_ids_fixed_kernel<IdT, 3, 2, OutT, kCarry, kIdx>;
    if (N == 3 && hpn == 4) return row_ids_fixed_kernel<IdT, 3, 4, OutT, kCarry, kIdx>;
    if (N == 4 && hpn == 4) return row_ids_fixed_kernel<IdT, 4, 4, OutT, kCarry, kIdx>;
    return row_ids_fixed_kernel<IdT, 5, 8, OutT, kCarry, kIdx>;
}

template <typename IdT, typename OutT, bool kCarry>
KernelFn pick_fixed(int N, int hpn, int mode) {
    if (mode == kIdxDecode) return pick_fixed<IdT, OutT, kCarry, kIdxDecode>(N, hpn);
    if (mode == kIdxCu) return pick_fixed<IdT, OutT, kCarry, kIdxCu>(N, hpn);
    return pick_fixed<IdT, OutT, kCarry, kIdxArrays>(N, hpn);
}

template <typename IdT, typename OutT>
KernelFn pick_fixed(int N, int hpn, bool carry, int mode) {
    return carry ? pick_fixed<IdT, OutT, true>(N, hpn, mode)
                 : pick_fixed<IdT, OutT, false>(N, hpn, mode);
}

}  // namespace

cudaError_t launch_row_ids_fixed(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                 cudaStream_t stream) {
    const bool carry = p.next_ctx != nullptr;
    const int mode = p.index_mode;
    KernelFn fn;
    if (p.out_bytes == 4)
        fn = id_bytes == 4 ? pick_fixed<int32_t, int32_t>(p.N, p.hpn, carry, mode)
                           : pick_fixed<int64_t, int32_t>(p.N, p.hpn, carry, mode);
    else
        fn = id_bytes == 4 ? pick_fixed<int32_t, int64_t>(p.N, p.hpn, carry, mode)
                           : pick_fixed<int64_t, int64_t>(p.N, p.hpn, carry, mode);
    return launch_fn(fn, p, cfg, stream);
}

}  // namespace ple
