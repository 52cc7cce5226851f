// Internal launch interface between the C ABI (ple_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ple {

// Tokens per warp tile of the row-id kernel (two per lane).
constexpr int kTileTokens = 64;
// Halo slots kept in front of each warp's staged ids (>= PLE_MAX_NGRAM - 1,
// even so the tile itself starts 16-byte aligned).
constexpr int kHaloSlots = 16;
// Upper bound on warps per thread block of the row-id kernel.
#ifndef PLE_MAX_WARPS
#define PLE_MAX_WARPS 4
#endif
constexpr int kMaxWarps = PLE_MAX_WARPS;
// Register cap for the fixed-shape kernel: the minimum resident blocks per SM
// passed to __launch_bounds__ (0 leaves the choice to the compiler).  Eight
// (64 registers a thread) measured best on GB300 across the large prefill and
// the mixed batch, int64 and int32 row ids alike: against the compiler's own
// budget the large prefill 30.2 -> 29.8 us (int64 row ids) and the mixed
// batch's int32 variant 12.8 -> 12.5 us; against nine blocks (56 registers)
// the large prefill's int32 variant 23.2 -> 22.7 us.
#ifndef PLE_FIXED_MIN_BLOCKS
#define PLE_FIXED_MIN_BLOCKS 8
#endif
constexpr int kFixedMinBlocks = PLE_FIXED_MIN_BLOCKS;
// Launch-shape target: thread blocks per SM the layer grouping aims for --
// 32 for int64 row ids (write-bound: smaller layer groups keep more
// independent stores in flight), 8 for int32 row ids (bound by instruction
// issue: larger groups share each token's window and cost fewer, longer
// blocks), 16 for the fused gather.  Measured on GB300: the large prefill's
// one-launch step 30.4 -> 30.0 us and the mixed batch's 18.3 -> 17.3 us at 32
// (against 16); int32 row ids of the large prefill 22.6 -> 21.9 us and of the
// mixed batch 13.6 -> 13.3 us at 8 (against 16; 5 was better for the large
// prefill, 21.6 us, but worse for the mixed batch, 14.6 us).
#ifndef PLE_BLOCKS_PER_SM
#define PLE_BLOCKS_PER_SM 8
#endif
#ifndef PLE_BLOCKS_PER_SM_I64
#define PLE_BLOCKS_PER_SM_I64 32
#endif
#ifndef PLE_BLOCKS_PER_SM_EMBED
#define PLE_BLOCKS_PER_SM_EMBED 16
#endif
constexpr int kTargetBlocksPerSm = PLE_BLOCKS_PER_SM;
constexpr int kTargetBlocksPerSmEmbed = PLE_BLOCKS_PER_SM_EMBED;
constexpr int kTargetBlocksPerSmI64 = PLE_BLOCKS_PER_SM_I64;

// A grid with fewer blocks than this many per SM (times the SM count) takes
// fewer warps per block, so that its warps spread over more SMs (0: never).
#ifndef PLE_SPREAD_BLOCKS_PER_SM
#define PLE_SPREAD_BLOCKS_PER_SM 1
#endif
constexpr int kSpreadBlocksPerSm = PLE_SPREAD_BLOCKS_PER_SM;
// Shared-memory budget for the per-head constants of one layer group.
constexpr int kConstBudgetBytes = 48 * 1024;
// Batches of at most this many row ids (T * H * L) take the small-batch
// kernel (one thread per row id); larger ones the tiled kernels.
#ifndef PLE_SMALL_MAX_ROWS
#define PLE_SMALL_MAX_ROWS 131072
#endif
constexpr int64_t kSmallMaxRows = PLE_SMALL_MAX_ROWS;
// Threads per block the small-batch kernel aims for (tokens x heads), and
// its hard maximum (one token of PLE_MAX_HEADS heads).
constexpr int kSmallBlockThreads = 128;
constexpr int kSmallMaxThreads = 256;

// How the kernels find each token's (request, offset):
//   kIdxArrays  read req[t], local[t] (an index built by ple_build_token_index)
//   kIdxDecode  a decode batch: req = t, local = 0, nothing read
//   kIdxCu      search cu_seqlens for the request owning t, local = t - start
enum IndexMode : int32_t { kIdxArrays = 0, kIdxDecode = 1, kIdxCu = 2 };

struct RowIdsParams {
    const void* ids;        // [T] int32 or int64
    const int32_t* req;     // [T]
    const int32_t* local;   // [T]
    const void* ctx;        // [B, N-1], dtype of ids
    const int64_t* mult;    // [L, N]
    const int64_t* vocab;   // [L, H]
    const int64_t* offsets; // [L, H]
    void* out;              // [L, T, H] int64 or int32 (out_bytes)
    int64_t T;
    int64_t boundary;
    int32_t B;
    int32_t N;
    int32_t hpn;
    int32_t H;
    int32_t L;
    int32_t group_layers;   // layers handled per thread block (grid.y groups)
    int32_t stage_pitch;    // row pitch (in int64) of the output staging tile
    int32_t ids_vec_ok;     // ids pointer is 16-byte aligned
    int32_t out_vec_ok;     // out pointer is 16-byte aligned
    int32_t index_mode;     // IndexMode
    int32_t out_bytes;      // 8: int64 row ids, 4: their low 32 bits
    const int32_t* cu;      // [B+1] cu_seqlens: kIdxCu and the context carry (NULL: none)
    void* next_ctx;         // [B, N-1] carried context out, dtype of ids (NULL: none)
    const void* heads;      // [L, H] prepared head constants (NULL: derive from vocab)
    uint32_t ones;          // 0xFFFFFFFF, opaque to the compiler (floormod_fast_alu)
};

// The table gather fused with the hash: table [L, rows, dim] bfloat16 bits,
// out [L, T, dim] float.
struct EmbedArgs {
    const uint16_t* table;
    int64_t rows;
    int32_t dim;
    float* out;
};

// Whether kernels are launched with programmatic stream serialization
// (process-wide, on unless turned off by ple_set_programmatic_launch).
bool programmatic_launch();

// Launches fn on stream and returns the launch's own status (the caller's
// pending CUDA error state is neither read nor cleared).  With programmatic
// stream serialization the launch may begin while the kernel before it in
// the stream drains: every kernel of this library waits for its predecessor
// grid before its first global memory access, so nothing is read early, and
// the launch overhead of back-to-back calls overlaps the kernel before.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool programmatic, Args... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = programmatic ? attr : nullptr;
    lc.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&lc, fn, args...);
}

struct RowIdsLaunch {
    dim3 grid;
    dim3 block;
    size_t smem_bytes;
    bool small;  // the small-batch kernel (else a tiled one)
};

// Per-device facts the launch configuration depends on, cached per device.
struct DeviceFacts {
    int sm_count;
    int max_smem_optin;
};

cudaError_t device_facts(DeviceFacts* out);

// Chooses grid/block/shared memory and fills p.group_layers / p.stage_pitch.
// runtime_layout: size the shared memory for the runtime-shape kernel's
// staging whatever the shape (the fused table gather uses that layout).
RowIdsLaunch plan_row_ids(RowIdsParams& p, const DeviceFacts& dev, bool runtime_layout = false);
cudaError_t launch_row_ids(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                           cudaStream_t stream);
// The tuned (ngram_size, heads_per_ngram) pairs of the fixed-shape kernel.
bool shape_is_fixed(int N, int hpn);
// Tuned shapes hashed by the head-lane kernel (ple_rowids_headlane.cu): the
// choice, whether its heads' constants are shared by the block (in shared
// memory, ahead of the per-warp memory), its per-warp shared memory, tile and
// launch.
bool uses_headlane_kernel(const RowIdsParams& p);
bool headlane_shared_constants(const RowIdsParams& p);
size_t headlane_smem_bytes(int N, int warps);
int headlane_tile_tokens();
cudaError_t launch_row_ids_headlane(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                    cudaStream_t stream);
cudaError_t launch_row_ids_fixed(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                 cudaStream_t stream);
// The small-batch kernel: whether a batch is small enough, its launch shape,
// its launch.
bool small_batch_fits(const RowIdsParams& p);
RowIdsLaunch plan_small(RowIdsParams& p);
cudaError_t launch_row_ids_small(const RowIdsParams& p, int id_bytes, const RowIdsLaunch& cfg,
                                 cudaStream_t stream);

cudaError_t launch_row_embed(const RowIdsParams& p, const EmbedArgs& e, int id_bytes,
                             const RowIdsLaunch& cfg, cudaStream_t stream);

cudaError_t launch_token_index(const int32_t* cu, int32_t B, int64_t T, int32_t is_decode,
                               int32_t* req, int32_t* local, const DeviceFacts& dev,
                               cudaStream_t stream);

cudaError_t launch_shard_inputs(const void* ids, int id_bytes, const int32_t* cu,
                                const void* ctx, int32_t B, int64_t T, int32_t C,
                                int64_t tok_begin, int64_t tok_end, int32_t req_begin,
                                int32_t req_count, int32_t* shard_cu, void* shard_ctx,
                                cudaStream_t stream);

cudaError_t launch_validate_index(const int32_t* cu, int32_t B, int64_t T, int32_t is_decode,
                                  const int32_t* req, const int32_t* local, int64_t* first_bad,
                                  const DeviceFacts& dev, cudaStream_t stream);

cudaError_t launch_prepare_heads(const int64_t* vocab, const int64_t* offsets, int64_t n,
                                 void* heads, const DeviceFacts& dev, cudaStream_t stream);

cudaError_t launch_selftest_floor_mod(const int64_t* x, const int64_t* v, int64_t n,
                                      int64_t* out_fast, int64_t* out_ref, const DeviceFacts& dev,
                                      cudaStream_t stream);

}  // namespace ple
