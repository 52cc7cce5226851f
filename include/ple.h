/*
 * ple.h -- C ABI of the GB300 (sm_103a) PLE n-gram row-id hash library.
 *
 * The operation is the per-layer-embedding (PLE) n-gram row-id hash of
 * FreeToken PR #338, "perf(ple): fuse the n-gram row-id hash into one Triton
 * kernel" (section "What"): for every token of a ragged decode or prefill
 * batch, find the token's n-gram window across its request's carried
 * context, mark which shifts cross a boundary token, and hash each n-gram
 * order with multiply / XOR into table row ids with a floored remainder plus
 * a per-head offset.
 *
 * Conventions shared by every entry point:
 *   - Every array argument is a DEVICE pointer (cudaMalloc'd or otherwise
 *     device-accessible) owned by the caller, except in ple_shard_plan,
 *     which is host code on host arrays.  The library allocates nothing,
 *     keeps no per-call state, never reads device data on the host and never
 *     synchronises.  Inputs are read-only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  All work is enqueued on it; the calls return before it runs.
 *     The calls are safe to capture in a CUDA graph provided one call of the
 *     same kind was made on the device before capture (the first call on a
 *     device sets kernel attributes).
 *   - Every argument check is done on the host from the scalar arguments and
 *     pointer values only.  On any error nothing is launched and no output
 *     is written.  A launch failure is reported as PLE_ERR_CUDA; the CUDA
 *     error code is then available from ple_last_cuda_error().
 *   - Pointers must be aligned to their element size (4 bytes for int32
 *     arrays, 8 for int64 arrays); 16-byte alignment is not required except
 *     where an entry point says so (prepared head constants, the gather's
 *     table and output).
 *   - All integer arithmetic is int64 with two's-complement wrap-around, as
 *     torch's int64 tensor ops do.
 */
#ifndef PLE_H_
#define PLE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PLE_OK = 0,
    PLE_ERR_NULL = 1,           /* a required pointer is NULL */
    PLE_ERR_SIZE = 2,           /* a size or count is out of the supported range */
    PLE_ERR_GEOMETRY_CTX = 3,   /* ctx_len != ngram_size - 1 */
    PLE_ERR_GEOMETRY_HEADS = 4, /* num_heads != (ngram_size - 1) * heads_per_ngram */
    PLE_ERR_DTYPE = 5,          /* id_dtype is neither PLE_I32 nor PLE_I64 */
    PLE_ERR_ALIGN = 6,          /* a pointer is not aligned to its element size */
    PLE_ERR_CUDA = 7            /* a CUDA call failed; see ple_last_cuda_error() */
} ple_status;

typedef enum { PLE_I32 = 0, PLE_I64 = 1 } ple_id_dtype;

#define PLE_MAX_NGRAM 16   /* largest supported ngram_size */
#define PLE_MAX_HEADS 256  /* largest supported heads per layer */
#define PLE_MAX_EMBED_DIM 65536  /* largest supported table row width */
#define PLE_HEAD_BYTES 48  /* bytes of one head's prepared constants */

/*
 * ple_build_token_index -- per-token (request, offset) index.
 *
 * Defined by the second observation of section "What" (token t belongs to
 * request req[t] at intra-request offset local[t]) and by the index note of
 * section "Why it is safe" (a decode is one token per request at offset 0;
 * a decode of B requests and a prefill of one B-token request have the same
 * shape and opposite meaning).
 *
 *   cu_seqlens    [num_requests + 1] int32, device.  Request r owns tokens
 *                 cu_seqlens[r] <= t < cu_seqlens[r+1].  Must be
 *                 non-decreasing with cu_seqlens[0] = 0 and
 *                 cu_seqlens[num_requests] = num_tokens (device data, not
 *                 checked; other contents give unspecified but in-range
 *                 req values).  Ignored (may be NULL) when is_decode != 0.
 *   num_requests  B >= 1 when num_tokens > 0.  For a decode, B == num_tokens.
 *   num_tokens    T, 0 <= T <= INT32_MAX.  T == 0 returns PLE_OK, no launch.
 *   is_decode     non-zero: req[t] = t, local[t] = 0.
 *                 zero: req[t] = r with cu_seqlens[r] <= t < cu_seqlens[r+1]
 *                 (empty requests own no token), local[t] = t - cu_seqlens[r].
 *   req, local    [T] int32 outputs, device.
 *
 * Errors: PLE_ERR_NULL, PLE_ERR_SIZE, PLE_ERR_ALIGN, PLE_ERR_CUDA.
 * One kernel launch.
 */
ple_status ple_build_token_index(const int32_t* cu_seqlens, int32_t num_requests,
                                 int64_t num_tokens, int32_t is_decode, int32_t* req,
                                 int32_t* local, void* stream);

/*
 * ple_row_ids -- the PLE n-gram row-id hash, all layers in one launch.
 *
 * Defined by section "What" of the page (packed window, boundary scan,
 * per-n-gram multiply / XOR / remainder / offset; the boundary walk of the
 * first observation and the window addressing of the second) and by section
 * "Why it is safe" (torch.remainder's floored sign rule; the two geometry
 * preconditions, raised rather than asserted).  With N = ngram_size,
 * hpn = heads_per_ngram, H = (N-1)*hpn, C = N-1, p = C + local[t]:
 *
 *   W(t,s)  = input_ids[t-s]                        if local[t] >= s
 *           = ngram_context[req[t]][C + local[t] - s] otherwise
 *   shift s is valid iff no boundary id is among W(t,1..s) (the token itself
 *   is not checked; s = 0 is always valid);
 *   V(t,s)  = W(t,s) if shift s is valid, else boundary_id;
 *   for n = 2..N and j < hpn, head h = (n-2)*hpn + j:
 *     mix   = XOR over s < n of V(t,s) * layer_multipliers[l][s]   (wrapping)
 *     out[l][t][h] = floormod(mix, vocab_sizes[l][h]) + offsets[l][h]
 *   where floormod takes the divisor's sign (torch.remainder).
 *
 *   input_ids           [T] int32 or int64 (id_dtype), device.  int32 ids are
 *                       sign-extended to int64.
 *   id_dtype            PLE_I32 or PLE_I64; also the dtype of ngram_context.
 *   num_tokens          T, 0 <= T <= INT32_MAX.  T == 0: PLE_OK, no launch.
 *   req, local          [T] int32, device, e.g. from ple_build_token_index.
 *                       Preconditions (device data, not checked): 0 <= req <
 *                       B, and the tokens of a request are contiguous and in
 *                       order, so 0 <= local[t] <= t.  Values outside these
 *                       ranges are clamped into them: the kernel never reads
 *                       out of bounds, but such rows are unspecified.
 *                       Both NULL: a decode batch (requires B == T), each
 *                       token its own request at offset 0 -- the index is
 *                       neither built nor read (one launch per step).
 *   ngram_context       [B, ctx_len], dtype id_dtype, device: each request's
 *                       last ctx_len ids before this batch, oldest first.
 *   num_requests        B >= 1 when T > 0.
 *   ctx_len             must equal N - 1 (else PLE_ERR_GEOMETRY_CTX).
 *   layer_multipliers   [L, N] int64, device; M[l][s] multiplies the id s
 *                       places left of the token (s = 0: the token).
 *   vocab_sizes         [L, H] int64, device.  Any non-zero value; negative
 *                       sizes follow torch.remainder (result in (v, 0]).  A
 *                       zero size yields the head's offset (torch raises).
 *   offsets             [L, H] int64, device.
 *   num_heads           H; must equal (N-1)*hpn (else PLE_ERR_GEOMETRY_HEADS);
 *                       at most PLE_MAX_HEADS.
 *   ngram_size          N, 2 <= N <= PLE_MAX_NGRAM.
 *   heads_per_ngram     hpn >= 1.
 *   num_layers          L >= 1.  A per-layer call passes M + l*N,
 *                       vocab_sizes + l*H, offsets + l*H and L = 1.
 *   boundary_id         b, the boundary (eos) token id.
 *   out                 [L, T, H] int64, device; every element is written.
 *
 * Errors: PLE_ERR_SIZE, PLE_ERR_GEOMETRY_CTX, PLE_ERR_GEOMETRY_HEADS (checked
 * in that order, before anything else), then PLE_ERR_NULL (one of req /
 * local NULL, or any other pointer), PLE_ERR_SIZE (both NULL with B != T),
 * PLE_ERR_DTYPE, PLE_ERR_ALIGN, PLE_ERR_CUDA.  PLE_ERR_SIZE also when the
 * output's byte count, L * T * H * 8, would not fit in int64.
 * One kernel launch; no host reads; the grid depends only on the sizes, the
 * way the index is given and the device (so a captured graph replays it).
 * Batches of at most ple_small_batch_max_rows() row ids (T * H * L) run the
 * small-batch kernel, one thread per row id; larger ones the tiled kernels.
 * The row ids are the same either way.
 */
ple_status ple_row_ids(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                       const int32_t* req, const int32_t* local, const void* ngram_context,
                       int32_t num_requests, int32_t ctx_len, const int64_t* layer_multipliers,
                       const int64_t* vocab_sizes, const int64_t* offsets, int32_t num_heads,
                       int32_t ngram_size, int32_t heads_per_ngram, int32_t num_layers,
                       int64_t boundary_id, int64_t* out, void* stream);

/*
 * ple_row_ids_i32 -- ple_row_ids with int32 row ids.
 *
 * The same operation, arguments, checks and launch as ple_row_ids, except
 * that `out` is [L, T, H] int32 (4-byte aligned) and receives the low 32
 * bits of each int64 row id (two's complement, as torch converts int64 to
 * int32).  Row ids below 2^31 -- every table whose offsets plus vocab sizes
 * stay below 2^31 -- are unchanged; the output bytes halve.  This is an
 * opt-in variant: the page's row ids are int64 (section "What").
 */
ple_status ple_row_ids_i32(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                           const int32_t* req, const int32_t* local, const void* ngram_context,
                           int32_t num_requests, int32_t ctx_len,
                           const int64_t* layer_multipliers, const int64_t* vocab_sizes,
                           const int64_t* offsets, int32_t num_heads, int32_t ngram_size,
                           int32_t heads_per_ngram, int32_t num_layers, int64_t boundary_id,
                           int32_t* out, void* stream);

/*
 * ple_row_ids_ex -- ple_row_ids with the output dtype chosen, the token
 * index optionally found in the kernel from cu_seqlens, the request contexts
 * carried to the next call in the same launch, and optionally the head
 * constants prepared by ple_prepare_heads.
 *
 * With req = local = NULL and cu_seqlens given, the kernel finds each
 * token's request itself: the request r with cu_seqlens[r] <= t <
 * cu_seqlens[r+1] (a binary search; empty requests own no token), at offset
 * t - cu_seqlens[r] -- the index ple_build_token_index would build, so a
 * prefill step is one launch and reads no index.  cu_seqlens must then
 * describe the batch as ple_build_token_index requires (device data, not
 * checked; other contents give unspecified rows, never an out-of-bounds
 * access).
 *
 * The carried context is the state that section "What" (second observation)
 * reads through ngram_context: each request's last ngram_size-1 ids before
 * the batch.  After this call, next_context[r] holds the last ctx_len ids of
 * (ngram_context[r], then request r's tokens of this batch), oldest first --
 * what the request's next prefill chunk or decode step passes as its
 * ngram_context.  A request with no token in the batch keeps its row.
 *
 *   all arguments up to boundary_id: as ple_row_ids, except that req = local
 *                 = NULL with cu_seqlens given takes any B >= 1 (above).  With
 *                 req = local = NULL and no cu_seqlens: a decode batch, as in
 *                 ple_row_ids.
 *   out           [L, T, H] int64 (out_dtype PLE_I64) or int32 (PLE_I32, the
 *                 low 32 bits as in ple_row_ids_i32), aligned to its element.
 *   out_dtype     PLE_I64 or PLE_I32 (else PLE_ERR_DTYPE).
 *   cu_seqlens    [B+1] int32, device, 4-byte aligned: the batch layout.
 *                 With req and local: the layout the index was built from,
 *                 required with next_context and otherwise not read.  Without
 *                 them: the layout the kernel searches (above); NULL there
 *                 means a decode batch, where every token ends its request.
 *   next_context  optional [B, ctx_len] output, dtype id_dtype, device; NULL
 *                 for no carry.  Must not overlap ngram_context (the kernel
 *                 reads every context row while it writes).
 *   heads         optional, device, 16-byte aligned: the constants
 *                 ple_prepare_heads wrote for these vocab_sizes and offsets.
 *                 When given, vocab_sizes and offsets are not read (they may
 *                 be NULL); NULL derives the constants in the call.
 *
 * Errors: as ple_row_ids, plus PLE_ERR_DTYPE for out_dtype, PLE_ERR_NULL
 * for a carry with req and local but without cu_seqlens, and PLE_ERR_ALIGN
 * for heads not 16-byte aligned or cu_seqlens not 4-byte aligned.
 */
ple_status ple_row_ids_ex(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                          const int32_t* req, const int32_t* local, const void* ngram_context,
                          int32_t num_requests, int32_t ctx_len, const int64_t* layer_multipliers,
                          const int64_t* vocab_sizes, const int64_t* offsets, int32_t num_heads,
                          int32_t ngram_size, int32_t heads_per_ngram, int32_t num_layers,
                          int64_t boundary_id, void* out, int32_t out_dtype,
                          const int32_t* cu_seqlens, void* next_context, const void* heads,
                          void* stream);

/*
 * ple_prepare_heads -- each head's remainder constants, computed once.
 *
 * Every row id ends with floormod(mix, vocab_sizes[l][h]) + offsets[l][h]
 * (section "What"; the floored sign rule of section "Why it is safe").  The
 * kernels do that remainder with a few multiplies by a per-head reciprocal
 * (Barrett / Granlund-Montgomery), which costs one 64-bit division per head
 * to set up -- a step of its own on the critical path of a decode call.
 * vocab_sizes and offsets are model parameters, so a caller that hashes many
 * batches with the same ones can set the constants up once here and pass
 * them as `heads` to ple_row_ids_ex.  The row ids are the same either way.
 * No counterpart on the page: a library-side precomputation.
 *
 *   vocab_sizes, offsets  [L, H] int64, device, as ple_row_ids.
 *   num_layers, num_heads L >= 1, 1 <= H <= PLE_MAX_HEADS.
 *   heads                 output, device, L * H * PLE_HEAD_BYTES bytes, 16-byte
 *                         aligned; an opaque layout valid for these
 *                         parameters only (a later change to vocab_sizes or
 *                         offsets needs a new call).
 *
 * Errors: PLE_ERR_SIZE, PLE_ERR_NULL, PLE_ERR_ALIGN, PLE_ERR_CUDA.
 * One kernel launch (ordered after earlier work on the stream).
 */
ple_status ple_prepare_heads(const int64_t* vocab_sizes, const int64_t* offsets,
                             int32_t num_layers, int32_t num_heads, void* heads, void* stream);

/*
 * ple_row_embed -- the row ids' table gather, fused with the hash.
 *
 * The row ids of section "What" are table row ids; this call hashes them
 * exactly as ple_row_ids does and, without writing them, sums over heads the
 * rows of the layer's embedding table that they name:
 *   out[l][t][:] = sum over h of table[l][row(l,t,h)][:]
 * accumulated in fp32 in head order (h = 0 first); a row id outside
 * [0, table_rows) adds nothing.  One launch for every layer.
 *
 *   all arguments up to boundary_id: as ple_row_ids_ex (req = local = NULL:
 *                 the requests found from cu_seqlens when it is given, else
 *                 a decode batch).
 *   table         [L, table_rows, dim] bfloat16 (as raw 16-bit patterns),
 *                 device, 16-byte aligned; may be NULL when table_rows == 0.
 *   table_rows    V >= 0 rows per layer.
 *   dim           D, a multiple of 8 in [8, PLE_MAX_EMBED_DIM].
 *   out           [L, T, D] float, device, 16-byte aligned; every element is
 *                 written.
 *   cu_seqlens    optional [B+1] int32, device: with req = local = NULL, the
 *                 layout the kernel searches for each token's request (as in
 *                 ple_row_ids_ex); not read when req and local are given.
 *   heads         optional: constants from ple_prepare_heads, as in
 *                 ple_row_ids_ex (vocab_sizes and offsets may then be NULL).
 *
 * Errors: as ple_row_ids_ex, plus PLE_ERR_SIZE for dim / table_rows or an
 * output of more than INT64_MAX bytes (L * T * dim * 4), and
 * PLE_ERR_ALIGN for a table or out that is not 16-byte aligned.
 */
ple_status ple_row_embed(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                         const int32_t* req, const int32_t* local, const void* ngram_context,
                         int32_t num_requests, int32_t ctx_len, const int64_t* layer_multipliers,
                         const int64_t* vocab_sizes, const int64_t* offsets, int32_t num_heads,
                         int32_t ngram_size, int32_t heads_per_ngram, int32_t num_layers,
                         int64_t boundary_id, const void* table, int64_t table_rows, int32_t dim,
                         float* out, const int32_t* cu_seqlens, const void* heads,
                         void* stream);

/*
 * ple_shard_plan -- one rank's share of a batch split by token range (host
 * code, host arrays; no CUDA call).
 *
 * Tokens are independent once each knows its window, and a request cut in
 * the middle continues from a carried context row: the last ngram_size - 1
 * ids before the cut (section "What", second observation: the window of a
 * token near its request's start reaches into the carried context).  So a
 * batch splits across ranks by token range with no exchange: rank k of
 * world_size takes tokens [T*k/world, T*(k+1)/world) (integer division) and
 * the requests that own them, hashes them as a batch of its own (inputs from
 * ple_shard_inputs) and writes its own [L, token_end - token_begin, H] rows,
 * which equal rows token_begin..token_end-1 of every layer of the whole
 * batch.
 *
 *   cu_seqlens   [num_requests + 1] int32, HOST: the whole batch's
 *                (non-decreasing, cu_seqlens[0] = 0, last = num_tokens;
 *                checked here, since it is host data).  NULL for a decode
 *                batch (one token per request): then the rank's requests
 *                are its tokens.
 *   num_requests B >= 1; num_tokens T >= 0 (T == B for a decode).
 *   world_size   >= 1; rank in [0, world_size).
 *   token_begin, token_end        out: the rank's tokens [begin, end).
 *   request_begin, request_count  out: the requests owning them, a
 *                contiguous range (request_count is 0 when the rank has no
 *                token).  A request with no token that starts exactly at a
 *                cut belongs to no rank; any other empty request between the
 *                rank's first and last owner is included.
 *
 * Errors: PLE_ERR_NULL (an output pointer), PLE_ERR_SIZE (counts out of
 * range, or cu_seqlens not a valid prefix sum of num_tokens).
 */
ple_status ple_shard_plan(const int32_t* cu_seqlens, int32_t num_requests, int64_t num_tokens,
                          int32_t world_size, int32_t rank, int64_t* token_begin,
                          int64_t* token_end, int32_t* request_begin, int32_t* request_count);

/*
 * ple_shard_inputs -- the per-rank inputs of ple_shard_plan's split, built on
 * the device from the whole batch's device arrays (one launch, no host read).
 *
 *   input_ids, id_dtype   [num_tokens] the whole batch's ids, device.  The
 *                         rank's ids are input_ids + token_begin (no copy).
 *   cu_seqlens            [num_requests + 1] int32, device: the whole batch's.
 *   ngram_context         [num_requests, ctx_len], dtype of the ids, device.
 *   num_requests, num_tokens, ctx_len (= ngram_size - 1, 1..15): the whole
 *                         batch's.
 *   token_begin, token_end, request_begin, request_count: from
 *                         ple_shard_plan (request_count >= 1).
 *   shard_cu_seqlens      [request_count + 1] int32 out, device: the rank's
 *                         cu_seqlens, cu_seqlens[request_begin + j] -
 *                         token_begin clamped to [0, token_end - token_begin].
 *   shard_context         [request_count, ctx_len] out, device, dtype of the
 *                         ids: request request_begin + j's context row for
 *                         the rank's call -- for the first request, cut at
 *                         token_begin, the last ctx_len ids of (its context
 *                         row, its tokens before token_begin); for the others
 *                         their own context row.
 *
 * Device data outside these rules (malformed cu_seqlens) gives unspecified
 * outputs but never an out-of-bounds access: every index is clamped.
 * Errors: PLE_ERR_NULL, PLE_ERR_SIZE, PLE_ERR_DTYPE, PLE_ERR_ALIGN,
 * PLE_ERR_CUDA.  One kernel launch.
 */
ple_status ple_shard_inputs(const void* input_ids, int32_t id_dtype, const int32_t* cu_seqlens,
                            const void* ngram_context, int32_t num_requests, int64_t num_tokens,
                            int32_t ctx_len, int64_t token_begin, int64_t token_end,
                            int32_t request_begin, int32_t request_count,
                            int32_t* shard_cu_seqlens, void* shard_context, void* stream);

/*
 * ple_validate_index -- diagnostic: check the index preconditions on the
 * device.
 *
 * ple_row_ids documents device-data preconditions on req / local that the
 * host cannot check without reading device memory; the kernel clamps such
 * data into range but the rows are then unspecified.  This call checks them
 * against their definition (section "What", second observation; "Why it is
 * safe", the decode rule): req[t] = r with cu_seqlens[r] <= t <
 * cu_seqlens[r+1] and local[t] = t - cu_seqlens[r], or req[t] = t and
 * local[t] = 0 for a decode.
 *
 *   cu_seqlens, num_requests, num_tokens, is_decode: as ple_build_token_index.
 *   req, local   [T] int32, device: the index to check.
 *   first_bad    one int64, device, 8-byte aligned.  The caller stores a
 *                value >= T there before the call; the call lowers it to the
 *                first token whose (req, local) is wrong and leaves it alone
 *                when every token is right.  Read it after the stream runs.
 *
 * Errors: PLE_ERR_NULL, PLE_ERR_SIZE, PLE_ERR_ALIGN, PLE_ERR_CUDA.
 */
ple_status ple_validate_index(const int32_t* cu_seqlens, int32_t num_requests,
                              int64_t num_tokens, int32_t is_decode, const int32_t* req,
                              const int32_t* local, int64_t* first_bad, void* stream);

/*
 * ple_selftest_floor_mod -- diagnostic: the library's invariant-divisor
 * floored remainder next to one computed with CUDA's own % operator.
 *
 * Section "Why it is safe" states that torch.remainder is floored while a
 * plain % truncates, so the kernel fixes the sign explicitly.  The row-id
 * kernel computes floormod(x, v) with a per-divisor reciprocal (Barrett
 * reduction) instead of %; this entry point exposes that routine so tests
 * can compare it, element by element, with CUDA's % plus the sign fix.
 *
 *   x, v        [n] int64, device (v may be anything; for v == 0 both
 *               outputs are 0).
 *   out_fast    [n] int64, device: the library's routine.
 *   out_ref     [n] int64, device: CUDA's % followed by the sign fix.
 *
 * Errors: PLE_ERR_NULL, PLE_ERR_SIZE (n < 0), PLE_ERR_ALIGN, PLE_ERR_CUDA.
 */
ple_status ple_selftest_floor_mod(const int64_t* x, const int64_t* v, int64_t n,
                                  int64_t* out_fast, int64_t* out_ref, void* stream);

/* The largest batch, in row ids (T * H * L, with L <= 65535), that the
 * row-id entry points hash with the small-batch kernel: latency-bound
 * decode steps and short prefills, one thread per row id, no block barrier.
 * A library tuning constant with no counterpart on the page; the row ids do
 * not depend on it. */
int64_t ple_small_batch_max_rows(void);

/*
 * ple_set_programmatic_launch -- process-wide switch for programmatic
 * dependent launch (on by default); returns the previous setting (1 or 0).
 *
 * Launch behaviour only, with no counterpart on the page: the row ids do not
 * depend on it.  When on, every kernel of this library is launched with
 * programmatic stream serialization and waits for the preceding grid in the
 * stream to complete before its first global memory access; so the launch of
 * one call overlaps the kernel before it (back-to-back calls, or the token
 * index build, which lets its dependent start at once, followed by the
 * row-id hash), and no memory is read early.
 * Off: every launch is an ordinary stream-ordered launch, so each call's
 * device time stands alone (for example, to time one call without overlap).
 * Takes effect for launches issued after it returns; safe from any thread.
 */
int32_t ple_set_programmatic_launch(int32_t enabled);

/* Static, NUL-terminated description of a status code ("unknown status"
 * for values outside ple_status). */
const char* ple_status_string(int32_t status);

/* The CUDA error code (a cudaError_t value) behind the last PLE_ERR_CUDA
 * returned on the calling thread, or 0. */
int32_t ple_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PLE_H_ */
