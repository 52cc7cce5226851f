// The PLE table gather fused with the n-gram row-id hash, on sm_103a.
//
// The row ids of FreeToken PR #338 ("perf(ple): fuse the n-gram row-id hash
// into one Triton kernel", section "What") are table row ids; their consumer
// gathers the named rows of the layer's embedding table.  This kernel hashes
// the row ids exactly as the row-id kernels do (shared code in
// ple_rowids_common.cuh) but keeps them in shared memory and, instead of
// writing them, sums over heads the table rows they name:
//
//   emb[l][t][:] = sum_h table[l][row(l,t,h)][:]       (fp32, head order)
//
// with table [L, V, D] bfloat16 and a row id outside [0, V) adding nothing.
// The work is an HBM gather: each (token, layer) reads H rows of 2*D bytes at
// random and writes 4*D bytes.  Each lane owns one 16-byte slice (8 values)
// of a row, so a warp reads a 512-byte row (D = 256) in one instruction;
// eight heads' slices are loaded before they are accumulated, so every lane
// keeps up to eight independent 16-byte loads in flight.  Narrower rows put
// several tokens in one warp pass; wider rows loop over slices.
#include "ple_rowids_common.cuh"

namespace ple {
namespace {

// Accumulate eight bfloat16 values (a 16-byte slice, element 8c + k in half
// k of the little-endian words) into fp32: bf16 bits are the top half of an
// IEEE float, so widening is a shift.
__device__ __forceinline__ void accumulate8(float (&acc)[8], uint4 v) {
    acc[0] += __uint_as_float(v.x << 16);
    acc[1] += __uint_as_float(v.x & 0xFFFF0000u);
    acc[2] += __uint_as_float(v.y << 16);
    acc[3] += __uint_as_float(v.y & 0xFFFF0000u);
    acc[4] += __uint_as_float(v.z << 16);
    acc[5] += __uint_as_float(v.z & 0xFFFF0000u);
    acc[6] += __uint_as_float(v.w << 16);
    acc[7] += __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 load_slice(const uint4* __restrict__ tab, int64_t row, int64_t V,
                                            int slices, int c) {
    // out-of-range row ids add nothing: a zero slice (bf16 +0)
    if ((uint64_t)row >= (uint64_t)V) return make_uint4(0u, 0u, 0u, 0u);
    return __ldg(tab + row * slices + c);
}

// Sum the table rows named by one token's H staged row ids, for slice c:
// eight heads' loads are issued before any of them is accumulated (then
// four, then one at a time), so a lane keeps up to eight 16-byte loads in
// flight; the sum stays in head order.
__device__ __forceinline__ void gather_token(const int64_t* __restrict__ rows, int H,
                                             const uint4* __restrict__ tab, int64_t V,
                                             int slices, int c, float* __restrict__ dst) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int h = 0;
    for (; h + 8 <= H; h += 8) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = load_slice(tab, rows[h + k], V, slices, c);
#pragma unroll
        for (int k = 0; k < 8; ++k) accumulate8(acc, v[k]);
    }
    for (; h + 4 <= H; h += 4) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = load_slice(tab, rows[h + k], V, slices, c);
#pragma unroll
        for (int k = 0; k < 4; ++k) accumulate8(acc, v[k]);
    }
    for (; h < H; ++h) accumulate8(acc, load_slice(tab, rows[h], V, slices, c));
    float4* o = reinterpret_cast<float4*>(dst + 8 * c);
    __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
    __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
}

// The gather's rate depends on how many table loads are in flight, which
// the register budget decides: eight loads a lane under a budget of seven
// resident blocks a SM (72 registers) measured best on GB300 (large prefill,
// D = 256: 1.93 ms a call, against 1.97 at eight blocks, 2.03 at six, and
// 2.12 for four loads a lane with the compiler's own budget).  The index
// mode is compile-time, as in the row-id kernels.
constexpr int kEmbedMinBlocks = 7;

template <typename IdT, int NT, int kIdx>
__global__ void __launch_bounds__(kMaxWarps * 32, kEmbedMinBlocks)
row_embed_kernel(const RowIdsParams p, const EmbedArgs e) {
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

    // gather walk: 16-byte slices per row; several tokens per warp pass when
    // a row has fewer than 32 slices
    const int slices = e.dim >> 3;
    const int per_pass = slices >= 32 ? 1 : 32 / slices;
    const int sub = slices >= 32 ? 0 : lane / slices;
    const int c0 = slices >= 32 ? lane : lane % slices;
    const bool lane_on = sub < per_pass;

#pragma unroll 1
    for (int u = 0; u < kTileTokens / 32; ++u) {
        const int nsub = min(32, ntile - 32 * u);
        if (nsub <= 0) break;
        int64_t V[NMAX];
        int32_t r, q;
        window<IdT, NMAX, NT, kIdx>(p, ids_s, t0, 32 * u + lane, lane < nsub, N, V, r, q);
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
            const uint4* tab = reinterpret_cast<const uint4*>(e.table) +
                               (int64_t)(l0 + l) * e.rows * slices;
            float* out = e.out + ((int64_t)(l0 + l) * p.T + t0 + 32 * u) * e.dim;
            if (lane_on) {
                for (int tb = 0; tb < nsub; tb += per_pass) {
                    const int tok = tb + sub;
                    if (tok >= nsub) break;
                    for (int c = c0; c < slices; c += 32)
                        gather_token(stage + tok * pitch, H, tab, e.rows, slices, c,
                                     out + (int64_t)tok * e.dim);
                }
            }
            __syncwarp();
        }
    }
}

using EmbedFn = void (*)(const RowIdsParams, const EmbedArgs);

template <typename IdT, int kIdx>
EmbedFn pick_embed(int N) {
    switch (N) {
        case 3: return row_embed_kernel<IdT, 3, kIdx>;
        case 4: return row_embed_kernel<IdT, 4, kIdx>;
        case 5: return row_embed_kernel<IdT, 5, kIdx>;
        default: return row_embed_kernel<IdT, 0, kIdx>;
    }
}

template <typename IdT>
EmbedFn pick_embed(int N, int mode) {
    if (mode == kIdxDecode) return pick_embed<IdT, kIdxDecode>(N);
    if (mode == kIdxCu) return pick_embed<IdT, kIdxCu>(N);
    return pick_embed<IdT, kIdxArrays>(N);
}

}  // namespace

cudaError_t launch_row_embed(const RowIdsParams& p, const EmbedArgs& e, int id_bytes,
                             const RowIdsLaunch& cfg, cudaStream_t stream) {
    const EmbedFn fn = id_bytes == 4 ? pick_embed<int32_t>(p.N, p.index_mode)
                                     : pick_embed<int64_t>(p.N, p.index_mode);
    if (cfg.smem_bytes > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)cfg.smem_bytes);
        if (err != cudaSuccess) return err;
    }
    return launch_kernel(fn, cfg.grid, cfg.block, cfg.smem_bytes, stream, programmatic_launch(),
                         p, e);
}

}  // namespace ple
