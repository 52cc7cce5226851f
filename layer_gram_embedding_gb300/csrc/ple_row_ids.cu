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
//   - grid.x covers the tokens in warp tiles of 64; grid.y splits the layers
//     into groups so that even a small T fills the SMs.
//   - Block prologue: the group's per-head divisor constants (one reciprocal
//     per head, see ple_divmod.cuh) and multipliers go to shared memory.
//   - Each warp stages its tile's ids plus an ngram_size-1 halo in shared
//     memory (16-byte vector loads when aligned) and builds each token's
//     window V in registers with the carried boundary predicate.
//   - Fixed shapes (the tuned (ngram_size, heads_per_ngram) pairs, even
//     heads per order): each lane hashes two tokens per shared constant load,
//     stages 32-bit remainders as head pairs in rows of odd pitch (8-byte
//     stores hit 16 distinct bank pairs per half warp), and the readout walks
//     the tile in global order ([L, T, H]), adds each head's offset in
//     registers and stores 16 bytes per lane: a warp store covers 512
//     consecutive bytes.
//   - Any other shape: one token per lane, int64 rows staged with odd pitch,
//     8-byte readout.  Heads off the 32-bit fast path (vocab outside
//     (0, 2^29]) use the same int64 staging in either kernel.
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

// Per-block shared-memory layout, in order (all offsets 16-byte aligned):
//   head constants of the layer group, structure of arrays:
//     fast [G*H] uint4, off [G*H] int64 (padded to even), ext [G*H] uint4
//   multipliers [G*N] int64 (padded to even)
//   per warp: ids [kHaloSlots + kTileTokens] int64
//   per warp: staging, stage_bytes(...) bytes
struct SmemLayout {
    uint4* fast;
    int64_t* off;
    uint4* ext;
    int64_t* mul;
    int64_t* ids;
    unsigned char* stage;
};

__host__ __device__ constexpr size_t head_const_bytes(int heads) {
    return (size_t)heads * 16 + (size_t)((heads + 1) & ~1) * 8 + (size_t)heads * 16;
}

// Staging bytes per warp.  Fixed shapes (even heads_per_ngram): 64 rows of
// 32-bit remainders in 8-byte pairs, odd pitch (H/2 | 1) pairs, or 32 rows of
// int64 rows with odd pitch (H | 1) for heads off the fast path -- whichever
// is larger.  Runtime shapes: 32 rows of int64 with odd pitch.
__host__ __device__ constexpr size_t stage_bytes(int H, bool fixed_shape) {
    return fixed_shape ? ((size_t)64 * ((H / 2) | 1) * 8 > (size_t)32 * (H | 1) * 8
                              ? (size_t)64 * ((H / 2) | 1) * 8
                              : (size_t)32 * (H | 1) * 8)
                       : (size_t)32 * (H | 1) * 8;
}

__device__ __forceinline__ SmemLayout carve_smem(unsigned char* base, int G, int H, int N,
                                                 int nwarps) {
    SmemLayout s;
    const int gh = G * H;
    s.fast = reinterpret_cast<uint4*>(base);
    s.off = reinterpret_cast<int64_t*>(base + (size_t)gh * 16);
    s.ext = reinterpret_cast<uint4*>(base + (size_t)gh * 16 + (size_t)((gh + 1) & ~1) * 8);
    s.mul = reinterpret_cast<int64_t*>(base + head_const_bytes(gh));
    s.ids = s.mul + ((G * N + 1) & ~1);
    s.stage = reinterpret_cast<unsigned char*>(s.ids + nwarps * (kHaloSlots + kTileTokens));
    return s;
}

// Block prologue: the layer group's head constants and multipliers.
// Returns this thread's vote on whether every head takes the 32-bit fast
// path; the caller publishes the constants with __syncthreads_and once its
// own window loads are in flight, so the per-head divisions overlap them.
__device__ __forceinline__ int load_group_constants(const RowIdsParams& p, const SmemLayout& sm,
                                                    int l0, int gl, int H, int N) {
    int fast = 1;
    for (int i = threadIdx.x; i < gl * H; i += blockDim.x) {
        const int64_t k = (int64_t)l0 * H + i;
        const HeadConst c = make_head_const(p.vocab[k], p.offsets[k]);
        sm.fast[i] = c.fast;
        sm.off[i] = c.off;
        sm.ext[i] = c.ext;
        fast &= (c.ext.z == kHeadFast) ? 1 : 0;
    }
    for (int i = threadIdx.x; i < gl * N; i += blockDim.x) sm.mul[i] = p.mult[(int64_t)l0 * N + i];
    return fast;
}

// Programmatic dependent launch: the row-id kernel may be scheduled while
// the kernel before it in the stream drains, so it waits for that grid's
// completion (and memory) before its first global read.  Without the launch
// attribute this returns at once.
__device__ __forceinline__ void wait_prior_grid() { cudaGridDependencySynchronize(); }

// Stage a warp tile's ids (and the N-1 ids left of it) in shared memory.
template <typename IdT>
__device__ __forceinline__ void stage_ids(const RowIdsParams& p, int64_t* ids_s, int64_t t0,
                                          int ntile, int N, int lane) {
    const IdT* ids = static_cast<const IdT*>(p.ids);
    if (ntile == kTileTokens && p.ids_vec_ok) {
        load_tile_vec<IdT>(ids + t0, ids_s, lane);
    } else {
        for (int i = lane; i < ntile; i += 32) ids_s[i] = load_id<IdT>(ids, t0 + i);
    }
    if (lane < N - 1 && t0 - 1 - lane >= 0) ids_s[-1 - lane] = load_id<IdT>(ids, t0 - 1 - lane);
    __syncwarp();
}

// The shifted window V(t, 0..N-1) of tile token i with the carried boundary
// predicate.  Index data outside the addressable ranges is clamped.
template <typename IdT, int NMAX, int NT>
__device__ __forceinline__ void window(const RowIdsParams& p, const int64_t* ids_s, int64_t t0,
                                       int i, bool live, int N, int64_t (&V)[NMAX]) {
    const int64_t t = t0 + i;
    int32_t r = 0, q = 0;
    if (p.index_free) {
        // a decode batch without an index: every token is its own request
        r = (int32_t)t;
    } else if (live) {
        r = __ldg(p.req + t);
        q = __ldg(p.local + t);
    }
    r = min(max(r, 0), p.B - 1);
    q = (int32_t)min((int64_t)max(q, 0), t);
    V[0] = live ? ids_s[i] : 0;
    const IdT* crow = static_cast<const IdT*>(p.ctx) + (int64_t)r * (N - 1) + (N - 1) + q;
    bool valid = true;
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
        if (NT == 0 && s >= N) break;
        const int64_t w = (q >= s) ? ids_s[i - s] : load_id<IdT>(crow, -s);
        valid = valid && (w != p.boundary);
        V[s] = valid ? w : p.boundary;
    }
}

// Hash one layer for one token into its int64 staging row (8-byte stores).
template <int NMAX, int NT, bool kFast>
__device__ __forceinline__ void hash_layer(const int64_t (&V)[NMAX], int N, int hpn,
                                           const int64_t* __restrict__ ml,
                                           const uint4* __restrict__ hf,
                                           const int64_t* __restrict__ ho,
                                           const uint4* __restrict__ he,
                                           int64_t* __restrict__ srow) {
    uint64_t mix = (uint64_t)V[0] * (uint64_t)ml[0];
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
        if (NT == 0 && s >= N) break;
        // order n = s + 1 folds shifts 0..s
        mix ^= (uint64_t)V[s] * (uint64_t)ml[s];
        const OffsetBinary u = offset_binary(mix);
        const int h0 = (s - 1) * hpn;
#pragma unroll 4
        for (int j = 0; j < hpn; ++j) {
            const int h = h0 + j;
            srow[h] = kFast ? row_fast(u, hf[h], ho[h]) : row_general(u, hf[h], ho[h], he[h]);
        }
    }
}

// Runtime-shape readout of one staged half tile (nsub tokens x H int64, row
// pitch `pitch`): one element per lane per step in global order, incremental
// (row, column).  An int32 destination receives each row id's low 32 bits.
template <typename OutT>
__device__ __forceinline__ void readout_runtime(const int64_t* __restrict__ stage,
                                                OutT* __restrict__ dst, int lane, int nsub,
                                                int H, int pitch) {
    const int dq = 32 / H;
    const int dr = 32 % H;
    int qq = lane / H;
    int rr = lane % H;
    const int nel = nsub * H;
    for (int e = lane; e < nel; e += 32) {
        if constexpr (sizeof(OutT) == 8)
            __stcs(reinterpret_cast<long long*>(dst) + e, (long long)stage[qq * pitch + rr]);
        else
            __stcs(reinterpret_cast<int*>(dst) + e, (int)stage[qq * pitch + rr]);
        rr += dr;
        qq += dq;
        if (rr >= H) {
            rr -= H;
            ++qq;
        }
    }
}

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
    const SmemLayout sm = carve_smem(smem, G, H, N, nwarps);
    const int fast_vote = load_group_constants(p, sm, l0, gl, H, N);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kTileTokens;
    const int ntile = (int)max((int64_t)0, min((int64_t)kTileTokens, p.T - t0));
    int64_t* ids_s = sm.ids + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
    int64_t* stage = reinterpret_cast<int64_t*>(sm.stage + (size_t)warp * stage_bytes(H, false));
    if (ntile > 0) stage_ids<IdT>(p, ids_s, t0, ntile, N, lane);
    const bool all_fast = __syncthreads_and(fast_vote) != 0;
    if (ntile == 0) return;

#pragma unroll 1
    for (int u = 0; u < kTileTokens / 32; ++u) {
        const int nsub = min(32, ntile - 32 * u);
        if (nsub <= 0) break;
        int64_t V[NMAX];
        window<IdT, NMAX, NT>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, V);
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

// int32 row ids: four heads (two staged pairs) per 16-byte lane store; the
// offsets' low words are added in 32-bit arithmetic (the low 32 bits of the
// int64 row id).  K2 quads per token.
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

template <typename IdT, int NT, int HPT, typename OutT>
__global__ void __launch_bounds__(kMaxWarps * 32)
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
    const SmemLayout sm = carve_smem(smem, G, H, N, nwarps);
    const int fast_vote = load_group_constants(p, sm, l0, gl, H, N);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * nwarps + warp) * kTileTokens;
    const int ntile = (int)max((int64_t)0, min((int64_t)kTileTokens, p.T - t0));
    int64_t* ids_s = sm.ids + warp * (kHaloSlots + kTileTokens) + kHaloSlots;
    unsigned char* stage = sm.stage + (size_t)warp * stage_bytes(H, true);
    const int nA = min(32, ntile);
    const int nB = ntile - 32;  // tokens in the second half (may be <= 0)
    int64_t VA[N], VB[N];
    if (ntile > 0) {
        stage_ids<IdT>(p, ids_s, t0, ntile, N, lane);
        window<IdT, N, N>(p, ids_s, t0, lane, lane < nA, N, VA);
        window<IdT, N, N>(p, ids_s, t0, 32 + lane, lane < nB, N, VB);
    }
    const bool all_fast = __syncthreads_and(fast_vote) != 0;
    if (ntile == 0) return;

    if (!all_fast) {
        // some head of this group is off the fast path: int64 rows, 8-byte
        // readout, one half tile at a time
        int64_t* st = reinterpret_cast<int64_t*>(stage);
#pragma unroll 1
        for (int u = 0; u < 2; ++u) {
            const int nsub = u == 0 ? nA : nB;
            if (nsub <= 0) break;
#pragma unroll 1
            for (int l = 0; l < gl; ++l) {
                const int hb = l * H;
                hash_layer<N, N, false>(u == 0 ? VA : VB, N, HPT, sm.mul + l * N, sm.fast + hb,
                                        sm.off + hb, sm.ext + hb, st + lane * PG);
                __syncwarp();
                OutT* dst = static_cast<OutT*>(p.out) +
                            ((int64_t)(l0 + l) * p.T + t0 + 32 * u) * H;
                readout_runtime<OutT>(st, dst, lane, nsub, H, PG);
                __syncwarp();
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
    int soff[KU], stok[KU];
#pragma unroll
    for (int j = 0; j < KU; ++j) {
        const int cj = (32 * j) % KU;
        const bool carry = r0 + cj >= KU;
        stok[j] = q0 + (32 * j) / KU + (carry ? 1 : 0);
        soff[j] = stok[j] * P2 + U * (r0 + cj - (carry ? KU : 0));
    }
    const bool full = nA == 32 && nB == 32;
    const bool vec_out = p.out_vec_ok != 0;

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
                stAw[lane * P2 + h / 2] = make_uint2(floormod_fast(uA, c0), floormod_fast(uA, c1));
                stAw[(32 + lane) * P2 + h / 2] =
                    make_uint2(floormod_fast(uB, c0), floormod_fast(uB, c1));
            }
        }
        __syncwarp();
        OutT* dst = static_cast<OutT*>(p.out) + ((int64_t)(l0 + l) * p.T + t0) * H;
        if constexpr (U == 1) {
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
        } else {
            int4 offs[NU];
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                int col = r0 + k * GU;
                col = col >= KU ? col - KU : col;
                const int64_t* o = sm.off + l * H + 4 * col;
                offs[k] = make_int4((int)o[0], (int)o[1], (int)o[2], (int)o[3]);
            }
            int* d = reinterpret_cast<int*>(dst);
            if (full && vec_out) {
                readout_quads<KU, P2, NU, GU, true, true>(stA, d, lane, 32, soff, stok, offs);
                readout_quads<KU, P2, NU, GU, true, true>(stA + 32 * P2, d + 32 * H, lane, 32,
                                                         soff, stok, offs);
            } else if (vec_out) {
                readout_quads<KU, P2, NU, GU, true, false>(stA, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_quads<KU, P2, NU, GU, true, false>(stA + 32 * P2, d + 32 * H, lane,
                                                              nB, soff, stok, offs);
            } else {
                readout_quads<KU, P2, NU, GU, false, false>(stA, d, lane, nA, soff, stok, offs);
                if (nB > 0)
                    readout_quads<KU, P2, NU, GU, false, false>(stA + 32 * P2, d + 32 * H, lane,
                                                               nB, soff, stok, offs);
            }
        }
        __syncwarp();
    }
}

using KernelFn = void (*)(const RowIdsParams);

// Compile-time shapes: the PLE configurations this library is tuned for
// (ngram_size, heads_per_ngram); everything else runs the runtime-shape
// kernel for its ngram_size.
template <typename IdT, typename OutT>
KernelFn pick_kernel(int N, int hpn) {
    if (N == 3 && hpn == 2) return row_ids_fixed_kernel<IdT, 3, 2, OutT>;
    if (N == 3 && hpn == 4) return row_ids_fixed_kernel<IdT, 3, 4, OutT>;
    if (N == 4 && hpn == 4) return row_ids_fixed_kernel<IdT, 4, 4, OutT>;
    if (N == 5 && hpn == 8) return row_ids_fixed_kernel<IdT, 5, 8, OutT>;
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

bool shape_is_fixed(int N, int hpn) {
    return (N == 3 && (hpn == 2 || hpn == 4)) || (N == 4 && hpn == 4) || (N == 5 && hpn == 8);
}

cudaError_t launch_fn(KernelFn fn, const RowIdsParams& p, const RowIdsLaunch& cfg,
                      cudaStream_t stream) {
    if (cfg.smem_bytes > 48 * 1024) {
        // Opting in to more than 48 KB of dynamic shared memory is a function
        // attribute; setting it is idempotent and not a stream operation.
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    // programmatic dependent launch: the blocks may become resident while the
    // previous kernel in the stream (typically the token-index build) drains;
    // the kernel waits for it before reading anything
    cudaLaunchConfig_t lc = {};
    lc.gridDim = cfg.grid;
    lc.blockDim = cfg.block;
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, fn, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

RowIdsLaunch plan_row_ids(RowIdsParams& p, const DeviceFacts& dev) {
    RowIdsLaunch cfg;
    const int64_t tiles = (p.T + kTileTokens - 1) / kTileTokens;
    int warps = (int)(tiles < kMaxWarps ? tiles : kMaxWarps);
    const bool fixed_shape = shape_is_fixed(p.N, p.hpn);
    p.stage_pitch = p.H | 1;
    const size_t per_warp =
        (size_t)(kHaloSlots + kTileTokens) * 8 + stage_bytes(p.H, fixed_shape);

    // layer groups: split the layers until there are kTargetBlocksPerSm
    // blocks per SM, so the last wave is short even when T alone gives few
    // tiles; constants stay within their shared-memory budget
    int64_t blocks_x = (tiles + warps - 1) / warps;
    const int64_t target = kTargetBlocksPerSm * (int64_t)dev.sm_count;
    int64_t groups = (target + blocks_x - 1) / blocks_x;
    if (groups < 1) groups = 1;
    if (groups > p.L) groups = p.L;
    int G = (int)((p.L + groups - 1) / groups);
    const int g_cap = (int)(kConstBudgetBytes / head_const_bytes(p.H));
    if (G > g_cap) G = g_cap > 0 ? g_cap : 1;
    groups = (p.L + G - 1) / G;
    p.group_layers = G;

    const size_t fixed = head_const_bytes(G * p.H) + round_up((size_t)G * p.N, 2) * 8;
    while (warps > 1 && fixed + warps * per_warp > (size_t)dev.max_smem_optin) --warps;
    blocks_x = (tiles + warps - 1) / warps;
    cfg.grid = dim3((unsigned)blocks_x, (unsigned)groups, 1);
    cfg.block = dim3(32 * warps, 1, 1);
    cfg.smem_bytes = fixed + warps * per_warp;
    return cfg;
}

cudaError_t launch_row_ids(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                           cudaStream_t stream) {
    KernelFn fn;
    if (p.out_bytes == 4)
        fn = id_bytes == 4 ? pick_kernel<int32_t, int32_t>(p.N, p.hpn)
                           : pick_kernel<int64_t, int32_t>(p.N, p.hpn);
    else
        fn = id_bytes == 4 ? pick_kernel<int32_t, int64_t>(p.N, p.hpn)
                           : pick_kernel<int64_t, int64_t>(p.N, p.hpn);
    return launch_fn(fn, p, cfg, stream);
}

}  // namespace ple
