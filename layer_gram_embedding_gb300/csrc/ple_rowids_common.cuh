// The PLE n-gram row-id hash on sm_103a: device code shared by the fixed-shape
// kernel (ple_rowids_fixed.cu), the runtime-shape kernel
// (ple_rowids_runtime.cu), the small-batch kernel (ple_rowids_small.cu) and
// the fused table gather (ple_embed.cu).
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
//     per head, see ple_divmod.cuh, or loaded when prepared once) and
//     multipliers go to shared memory.
//   - Each warp finds its tokens' (request, offset) -- read from an index,
//     synthesised for a decode, or searched in cu_seqlens -- while its tile's
//     ids plus an ngram_size-1 halo load (16-byte vectors when aligned), then
//     stages the ids in shared memory and builds each token's window V in
//     registers with the carried boundary predicate.
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
#pragma once

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

// Per-block shared-memory layout, in order (all offsets 16-byte aligned):
//   head constants of the layer group, structure of arrays:
//     fast [G*H] uint4, off [G*H] int64 (padded to even), ext [G*H] uint4,
//     off32 [G*H] the offsets' low words (padded to a multiple of 4), read
//     four at a time by the int32 readout
//   multipliers [G*N] int64 (padded to even)
//   per warp: ids [kHaloSlots + kTileTokens] int64
//   per warp: staging, stage_bytes(...) bytes
struct SmemLayout {
    uint4* fast;
    int64_t* off;
    uint4* ext;
    int32_t* off32;
    int64_t* mul;
    int64_t* ids;
    unsigned char* stage;
};

__host__ __device__ constexpr size_t head_const_bytes(int heads) {
    return (size_t)heads * 16 + (size_t)((heads + 1) & ~1) * 8 + (size_t)heads * 16 +
           (size_t)((heads + 3) & ~3) * 4;
}

// Fixed shapes with more heads than this stage half as many tokens at a
// time (a 32-token half tile on the fast path, a 16-token quarter on the
// general one), so that shared memory does not cap the resident blocks.
constexpr int kSplitStageHeads = 16;

__host__ __device__ constexpr int fast_stage_rows(int H) { return H > kSplitStageHeads ? 32 : 64; }
// Tokens per warp tile of the fixed-shape kernel.  A split-staging shape
// hashes one 32-token half at a time anyway, so it takes 32-token tiles:
// twice the warp tiles for grids that are short of them (the 48-layer mixed
// batch has 128 tiles of 64), and in the cu_seqlens search mode a tile spans
// at most 32 requests, so it always takes the lane ranking.  Measured on
// GB300 for the mixed batch, with int64 row ids at 32 blocks per SM: 18.0 ->
// 16.6 us reading an index, 18.3 -> 17.3 us in the search mode.
__host__ __device__ constexpr int fixed_tile_tokens(int H) {
    return H > kSplitStageHeads ? 32 : kTileTokens;
}
__host__ __device__ constexpr int general_stage_rows(int H) {
    return H > kSplitStageHeads ? 16 : 32;
}

// Staging bytes per warp.  Fixed shapes (even heads_per_ngram): rows of
// 32-bit remainders in 8-byte pairs, odd pitch (H/2 | 1) pairs, or int64 rows
// with odd pitch (H | 1) for heads off the fast path -- whichever is larger
// (row counts above).  Runtime shapes: 32 rows of int64 with odd pitch.
__host__ __device__ constexpr size_t stage_bytes(int H, bool fixed_shape) {
    return fixed_shape
               ? ((size_t)fast_stage_rows(H) * ((H / 2) | 1) * 8 >
                          (size_t)general_stage_rows(H) * (H | 1) * 8
                      ? (size_t)fast_stage_rows(H) * ((H / 2) | 1) * 8
                      : (size_t)general_stage_rows(H) * (H | 1) * 8)
               : (size_t)32 * (H | 1) * 8;
}

__device__ __forceinline__ SmemLayout carve_smem(unsigned char* base, int G, int H, int N,
                                                 int nwarps) {
    SmemLayout s;
    const int gh = G * H;
    s.fast = reinterpret_cast<uint4*>(base);
    s.off = reinterpret_cast<int64_t*>(base + (size_t)gh * 16);
    s.ext = reinterpret_cast<uint4*>(base + (size_t)gh * 16 + (size_t)((gh + 1) & ~1) * 8);
    s.off32 = reinterpret_cast<int32_t*>(base + (size_t)gh * 32 + (size_t)((gh + 1) & ~1) * 8);
    s.mul = reinterpret_cast<int64_t*>(base + head_const_bytes(gh));
    s.ids = s.mul + ((G * N + 1) & ~1);
    s.stage = reinterpret_cast<unsigned char*>(s.ids + nwarps * (kHaloSlots + kTileTokens));
    return s;
}

// Block prologue: the layer group's head constants (prepared ones loaded,
// else one reciprocal per head) and multipliers.
// Returns this thread's vote on whether every head takes the 32-bit fast
// path; the caller publishes the constants with __syncthreads_and once its
// own window loads are in flight, so the per-head divisions overlap them.
__device__ __forceinline__ int load_group_constants(const RowIdsParams& p, const SmemLayout& sm,
                                                    int l0, int gl, int H, int N) {
    int fast = 1;
    for (int i = threadIdx.x; i < gl * H; i += blockDim.x) {
        const int64_t k = (int64_t)l0 * H + i;
        const HeadConst c = p.heads != nullptr ? load_head_const(p.heads, k)
                                               : make_head_const(p.vocab[k], p.offsets[k]);
        sm.fast[i] = c.fast;
        sm.off[i] = c.off;
        sm.ext[i] = c.ext;
        sm.off32[i] = (int32_t)c.off;
        fast &= (c.ext.z == kHeadFast) ? 1 : 0;
    }
    for (int i = threadIdx.x; i < gl * N; i += blockDim.x) sm.mul[i] = p.mult[(int64_t)l0 * N + i];
    return fast;
}

// Programmatic dependent launch: the row-id kernel may be scheduled while
// the kernel before it in the stream drains, so it waits for that grid's
// completion (and memory) before its first global read.  Without the launch
// attribute this returns at once.  (Triggering this kernel's own dependents
// as it starts, so that their blocks could take the slots its tail frees,
// measured no faster on GB300: back-to-back large prefills 29.66 -> 29.59 us,
// the 48-layer mixed batch 17.44 -> 17.61 us, decode B=1 in a graph 1.28 ->
// 1.35 us.)
__device__ __forceinline__ void wait_prior_grid() { cudaGridDependencySynchronize(); }

// A warp tile's ids (and the N-1 ids left of it) staged in shared memory, in
// two steps so that other loads can be in flight meanwhile: fetch_tile_ids
// issues the loads into registers (16-byte vectors when the tile is full and
// aligned: two int64 ids per lane, or four int32 ids on 16 lanes; else at
// most two per lane), put_tile_ids stores them.
struct TileIds {
    int64_t a, b, c, d, halo;
};

template <typename IdT>
__device__ __forceinline__ TileIds fetch_tile_ids(const RowIdsParams& p, int64_t t0, int ntile,
                                                  int N, int lane) {
    TileIds f = {0, 0, 0, 0, 0};
    const IdT* ids = static_cast<const IdT*>(p.ids);
    if (ntile == kTileTokens && p.ids_vec_ok) {
        if constexpr (sizeof(IdT) == 8) {
            const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(ids + t0) + lane);
            f.a = v.x;
            f.b = v.y;
        } else if (lane < 16) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(ids + t0) + lane);
            f.a = v.x;
            f.b = v.y;
            f.c = v.z;
            f.d = v.w;
        }
    } else {
        if (lane < ntile) f.a = load_id<IdT>(ids, t0 + lane);
        if (lane + 32 < ntile) f.b = load_id<IdT>(ids, t0 + 32 + lane);
    }
    if (lane < N - 1 && t0 - 1 - lane >= 0) f.halo = load_id<IdT>(ids, t0 - 1 - lane);
    return f;
}

template <typename IdT>
__device__ __forceinline__ void put_tile_ids(const RowIdsParams& p, const TileIds& f,
                                             int64_t* ids_s, int64_t t0, int ntile, int N,
                                             int lane) {
    if (ntile == kTileTokens && p.ids_vec_ok) {
        if constexpr (sizeof(IdT) == 8) {
            reinterpret_cast<longlong2*>(ids_s)[lane] = make_longlong2(f.a, f.b);
        } else if (lane < 16) {
            longlong2* d = reinterpret_cast<longlong2*>(ids_s) + 2 * lane;
            d[0] = make_longlong2(f.a, f.b);
            d[1] = make_longlong2(f.c, f.d);
        }
    } else {
        if (lane < ntile) ids_s[lane] = f.a;
        if (lane + 32 < ntile) ids_s[lane + 32] = f.b;
    }
    if (lane < N - 1 && t0 - 1 - lane >= 0) ids_s[-1 - lane] = f.halo;
    __syncwarp();
}

template <typename IdT>
__device__ __forceinline__ void stage_ids(const RowIdsParams& p, int64_t* ids_s, int64_t t0,
                                          int ntile, int N, int lane) {
    put_tile_ids<IdT>(p, fetch_tile_ids<IdT>(p, t0, ntile, N, lane), ids_s, t0, ntile, N, lane);
}

// The requests owning tokens t1 and t2 in the cu_seqlens search mode, found
// by the whole warp for warp-uniform t1, t2: a 32-way search, one probe per
// lane per round for each (two rounds up to 1024 requests), the two in
// lockstep.  For well-formed cu_seqlens the lanes whose probe is <= t form
// a prefix and the owner lies in the last such lane's segment; whatever the
// contents the probes stay in cu[0..B-1] and each range shrinks every round.
// Every lane of the warp must call it.
__device__ __forceinline__ void warp_owners(const RowIdsParams& p, int64_t t1, int64_t t2,
                                            int lane, int& r1, int& r2) {
    int lo1 = 0, hi1 = p.B, lo2 = 0, hi2 = p.B;  // the owners are in [lo, hi)
    while (hi1 - lo1 > 1 || hi2 - lo2 > 1) {
        const int step1 = (hi1 - lo1 + 31) >> 5;
        const int step2 = (hi2 - lo2 + 31) >> 5;
        const int k1 = lo1 + lane * step1;
        const int k2 = lo2 + lane * step2;
        const bool le1 = hi1 - lo1 > 1 && k1 < hi1 && (int64_t)__ldg(p.cu + k1) <= t1;
        const bool le2 = hi2 - lo2 > 1 && k2 < hi2 && (int64_t)__ldg(p.cu + k2) <= t2;
        const unsigned m1 = __ballot_sync(0xffffffffu, le1);
        const unsigned m2 = __ballot_sync(0xffffffffu, le2);
        if (hi1 - lo1 > 1) {
            lo1 += (m1 ? 31 - __clz((int)m1) : 0) * step1;
            hi1 = min(hi1, lo1 + step1);
        }
        if (hi2 - lo2 > 1) {
            lo2 += (m2 ? 31 - __clz((int)m2) : 0) * step2;
            hi2 = min(hi2, lo2 + step2);
        }
    }
    r1 = lo1;
    r2 = lo2;
}

// The owners of a lane's two tokens tA, tB of a tile whose requests are
// ra..rb with rb - ra <= 32: lane j holds the start cu[ra + 1 + j] of one of
// the tile's later requests (past rb: a sentinel above every token), and a
// token's owner is ra plus the number of those starts at or below it -- for
// well-formed cu_seqlens a prefix of the lanes, counted by a 5-step shuffle
// search with no memory round trip.  Whatever the contents, only cu[ra..rb]
// is read and the results are clamped as load_index clamps them.  Every lane
// of the warp must call it.
__device__ __forceinline__ void tile_owners(const RowIdsParams& p, int ra, int rb, int64_t tA,
                                            bool liveA, int64_t tB, bool liveB, int lane,
                                            int32_t& rA, int32_t& qA, int32_t& rB,
                                            int32_t& qB) {
    const int k = ra + 1 + lane;
    const int32_t s = k <= rb ? __ldg(p.cu + k) : INT32_MAX;
    const int32_t s0 = __ldg(p.cu + ra);
    int cA = 0, cB = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
        const int32_t vA = __shfl_sync(0xffffffffu, s, cA + step - 1);
        const int32_t vB = __shfl_sync(0xffffffffu, s, cB + step - 1);
        if ((int64_t)vA <= tA) cA += step;
        if ((int64_t)vB <= tB) cB += step;
    }
    const int32_t last = __shfl_sync(0xffffffffu, s, 31);
    if (cA == 31 && (int64_t)last <= tA) cA = 32;
    if (cB == 31 && (int64_t)last <= tB) cB = 32;
    const int32_t pA = __shfl_sync(0xffffffffu, s, max(cA - 1, 0));
    const int32_t pB = __shfl_sync(0xffffffffu, s, max(cB - 1, 0));
    const int64_t startA = cA ? pA : s0;
    const int64_t startB = cB ? pB : s0;
    rA = liveA ? min(max(ra + cA, 0), p.B - 1) : 0;
    rB = liveB ? min(max(ra + cB, 0), p.B - 1) : 0;
    qA = liveA ? (int32_t)min(max(tA - startA, (int64_t)0), tA) : 0;
    qB = liveB ? (int32_t)min(max(tB - startB, (int64_t)0), tB) : 0;
}

// The shifted window V(t, 0..N-1) of tile token i with the carried boundary
// predicate, in two steps so a kernel can issue the index loads early:
// load_index finds (req, local) -- read, synthesised for a decode, or
// searched in cu_seqlens -- and clamps index data outside the addressable
// ranges; window_at builds V.  The mode is a compile-time choice: a run-time
// branch here costs the large-prefill kernel about 3% (measured on GB300).
template <int kMode>
__device__ __forceinline__ void load_index(const RowIdsParams& p, int64_t t, bool live,
                                           int32_t& r_out, int32_t& q_out, int ra = 0,
                                           int rb = -1) {
    int32_t r = 0, q = 0;
    if (kMode == kIdxDecode) {
        // a decode batch without an index: every token is its own request
        r = (int32_t)t;
    } else if (kMode == kIdxCu) {
        if (live) {
            // the request owning t is the last r with cu[r] <= t (an empty
            // request shares its start with the next one), searched in
            // [ra, rb] (the whole batch by default; a tiled kernel passes the
            // owners of its tile's first and last tokens).  The search keeps
            // cu[lo] <= t < cu[hi] for well-formed cu_seqlens and reads only
            // cu[ra..rb] whatever the contents.
            int lo = ra, hi = (rb < 0 ? p.B - 1 : rb) + 1;
            int32_t start = __ldg(p.cu + lo);
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                const int32_t c = __ldg(p.cu + mid);
                if ((int64_t)c <= t) {
                    lo = mid;
                    start = c;
                } else {
                    hi = mid;
                }
            }
            r = lo;
            q = (int32_t)min(max(t - (int64_t)start, (int64_t)0), t);
        }
    } else if (live) {
        r = __ldg(p.req + t);
        q = __ldg(p.local + t);
    }
    r_out = min(max(r, 0), p.B - 1);
    q_out = (int32_t)min((int64_t)max(q, 0), t);
}

// The window of tile token i from its (clamped) request r and offset q.
template <typename IdT, int NMAX, int NT>
__device__ __forceinline__ void window_at(const RowIdsParams& p, const int64_t* ids_s, int i,
                                          bool live, int N, int32_t r, int32_t q,
                                          int64_t (&V)[NMAX]) {
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

template <typename IdT, int NMAX, int NT, int kMode>
__device__ __forceinline__ void window(const RowIdsParams& p, const int64_t* ids_s, int64_t t0,
                                       int i, bool live, int N, int64_t (&V)[NMAX],
                                       int32_t& r_out, int32_t& q_out) {
    load_index<kMode>(p, t0 + i, live, r_out, q_out);
    window_at<IdT, NMAX, NT>(p, ids_s, i, live, N, r_out, q_out, V);
}

// The context carry: the last token of each request writes the request's
// next ngram_context row, the last N-1 ids of (context row, this batch's
// tokens) = W(t, N-2), ..., W(t, 0), oldest first.  Without cu_seqlens
// (a decode without an index) every token is the last of its request.
template <typename IdT>
__device__ __forceinline__ void carry_context(const RowIdsParams& p, const int64_t* ids_s,
                                              int64_t t0, int i, bool live, int N, int32_t r,
                                              int32_t q) {
    if (!live) return;
    const int64_t t = t0 + i;
    if (p.cu != nullptr && t != (int64_t)__ldg(p.cu + r + 1) - 1) return;
    const IdT* crow = static_cast<const IdT*>(p.ctx) + (int64_t)r * (N - 1) + (N - 1) + q;
    IdT* dst = static_cast<IdT*>(p.next_ctx) + (int64_t)r * (N - 1);
    for (int c = 0; c < N - 1; ++c) {
        const int s = N - 2 - c;
        dst[c] = (q >= s) ? (IdT)ids_s[i - s] : crow[-s];
    }
}

// Requests with no token in this batch keep their context row.  Needs
// cu_seqlens; run by the blocks of the first layer group (any block shape).
template <typename IdT>
__device__ __forceinline__ void carry_empty_requests(const RowIdsParams& p, int N) {
    if (p.next_ctx == nullptr || p.cu == nullptr || blockIdx.y != 0) return;
    const int64_t nthreads = (int64_t)blockDim.x * blockDim.y * blockDim.z;
    const int64_t tid = threadIdx.x + (int64_t)blockDim.x * (threadIdx.y + blockDim.y * threadIdx.z);
    const int64_t stride = (int64_t)gridDim.x * nthreads;
    for (int64_t r = (int64_t)blockIdx.x * nthreads + tid; r < p.B; r += stride) {
        if (__ldg(p.cu + r) == __ldg(p.cu + r + 1)) {
            const IdT* src = static_cast<const IdT*>(p.ctx) + r * (N - 1);
            IdT* dst = static_cast<IdT*>(p.next_ctx) + r * (N - 1);
            for (int c = 0; c < N - 1; ++c) dst[c] = src[c];
        }
    }
}

// A warp tile's windows: token t0 + lane's in VA and, for 64-token tiles,
// token t0 + 32 + lane's in VB, with the carried boundary predicate.  The
// tile's ids are fetched, each token's request is found (read from the
// index, synthesised for a decode, or searched in cu_seqlens, per kIdx), the
// ids are staged in shared memory at ids_s (with their N-1 halo) and the
// windows built; with kCarry the first layer group's blocks also write the
// next context.  Every lane of the warp calls it, with ntile > 0.
template <typename IdT, int N, int kTile, int kIdx, bool kCarry>
__device__ __forceinline__ void tile_windows(const RowIdsParams& p, int64_t* ids_s, int64_t t0,
                                             int ntile, int lane, int64_t (&VA)[N],
                                             int64_t (&VB)[N]) {
    const int nA = min(32, ntile);
    const int nB = ntile - 32;  // tokens in the second half (may be <= 0)
    // the tile's ids are fetched into registers first and stored to
    // shared memory only after the index is found, so the ids loads and
    // the index loads (or the cu_seqlens search) are in flight together
    const TileIds fetched = fetch_tile_ids<IdT>(p, t0, ntile, N, lane);
    int32_t rA, qA, rB, qB;
    if constexpr (kIdx == kIdxCu) {
        // the requests of the tile's first and last tokens bound every
        // token's owner: with at most 32 requests between them the lanes
        // rank the requests' starts (no search at all inside one
        // request), else each lane searches between them
        int ra, rb;
        warp_owners(p, t0, t0 + ntile - 1, lane, ra, rb);
        if (ra == rb) {
            // the whole tile inside one request
            const int64_t start = __ldg(p.cu + ra);
            rA = lane < nA ? ra : 0;
            rB = lane < nB ? ra : 0;
            qA = lane < nA ? (int32_t)min(max(t0 + lane - start, (int64_t)0), t0 + lane) : 0;
            qB = lane < nB
                     ? (int32_t)min(max(t0 + 32 + lane - start, (int64_t)0), t0 + 32 + lane)
                     : 0;
        } else if (rb - ra <= 32) {
            tile_owners(p, ra, rb, t0 + lane, lane < nA, t0 + 32 + lane, lane < nB, lane, rA,
                        qA, rB, qB);
        } else {
            load_index<kIdx>(p, t0 + lane, lane < nA, rA, qA, ra, rb);
            load_index<kIdx>(p, t0 + 32 + lane, lane < nB, rB, qB, ra, rb);
        }
    } else {
        load_index<kIdx>(p, t0 + lane, lane < nA, rA, qA);
        load_index<kIdx>(p, t0 + 32 + lane, lane < nB, rB, qB);
    }
    put_tile_ids<IdT>(p, fetched, ids_s, t0, ntile, N, lane);
    window_at<IdT, N, N>(p, ids_s, lane, lane < nA, N, rA, qA, VA);
    if constexpr (kTile == 64) {
        window_at<IdT, N, N>(p, ids_s, 32 + lane, lane < nB, N, rB, qB, VB);
    } else {
#pragma unroll
        for (int s = 0; s < N; ++s) VB[s] = 0;
    }
    if (kCarry && blockIdx.y == 0) {
        carry_context<IdT>(p, ids_s, t0, lane, lane < nA, N, rA, qA);
        if constexpr (kTile == 64)
            carry_context<IdT>(p, ids_s, t0, 32 + lane, lane < nB, N, rB, qB);
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

using KernelFn = void (*)(const RowIdsParams);

// Launch (with programmatic stream serialization unless it is turned off:
// see launch_kernel).  Opting in to more than 48 KB of dynamic shared memory
// is a function attribute; setting it is idempotent and not a stream
// operation.
inline cudaError_t launch_fn(KernelFn fn, const RowIdsParams& p, const RowIdsLaunch& cfg,
                             cudaStream_t stream) {
    if (cfg.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cfg.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(fn, cfg.grid, cfg.block, cfg.smem_bytes, stream, programmatic_launch(),
                         p);
}

}  // namespace
}  // namespace ple
