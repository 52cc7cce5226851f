/*
 * Reference oracle for the PLE n-gram row-id hash.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, single-threaded CPU restatement of what the
 * method computes.  It exists to check the CUDA library bit for bit and must
 * never sit on a product path: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header or table
 * with the CUDA library.
 *
 * Source of the definition: FreeToken PR #338, "perf(ple): fuse the n-gram
 * row-id hash into one Triton kernel".
 *   - section "What", first paragraph: the PLE layer packs the ragged tokens
 *     into an eos-filled [B, ctx+max_len] window, runs a cummax boundary scan
 *     over the whole window, then a per-n-gram loop of multiply / XOR /
 *     remainder / offset produces [T, num_ngram_heads] table row ids.
 *   - section "What", first observation: shift s is valid at window
 *     position p iff p - s >= 0 and no boundary token lies in [p-s, p-1].
 *   - section "What", second observation: token t sits in request req[t] at
 *     offset local[t]; left of the window is the boundary token.
 *   - section "Why it is safe": torch.remainder is floored (the result takes
 *     the divisor's sign); the context holds ngram_size-1 ids and each n-gram
 *     order owns heads_per_ngram heads.
 *
 * Readings taken where the page is silent (the readings below):
 *   - an invalid shift hashes the boundary id in place of the window value
 *     (reading "A"); reading "B" (an invalid shift contributes nothing to the
 *     XOR) is kept behind the `invalid_as_zero` flag for comparison only;
 *   - multiplier M[l][s] multiplies the value s places to the left (s = 0 is
 *     the token itself); order n folds shifts 0..n-1 with XOR, no seed;
 *   - int64 products and sums wrap modulo 2^64 (two's complement);
 *   - heads are order-major: head h = (n-2)*heads_per_ngram + j;
 *   - int32 ids are sign-extended to int64 before anything else;
 *   - out is [L, T, H] with layer l's slice equal to a one-layer call.
 *
 * Parity status: every function here is pinned by the `-m "not gpu"` tests
 * (a hand-worked window, brute-force enumeration, invariants, a closed form
 * for ngram_size 2).  Against the original FreeToken implementation parity is
 * unpinned: the page prints no row-id value, so the two readings above that
 * change values (invalid-shift value, multiplier order) rest on the text.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1       /* null pointer or negative size */
#define ORC_ERR_GEOMETRY 2  /* ctx_len != N-1 or H != (N-1)*hpn */
#define ORC_ERR_INDEX 3     /* (req, local) does not describe a packed batch */
#define ORC_ERR_VOCAB 4     /* a vocab size of zero: torch.remainder raises */
#define ORC_ERR_ALLOC 5

/* torch int64 multiply: wraps modulo 2^64. */
static int64_t wrap_mul(int64_t a, int64_t b) {
    return (int64_t)((uint64_t)a * (uint64_t)b);
}

/* torch int64 add: wraps modulo 2^64. */
static int64_t wrap_add(int64_t a, int64_t b) {
    return (int64_t)((uint64_t)a + (uint64_t)b);
}

/* torch.remainder on int64: floored, the result has the sign of v.
 * C's % truncates toward zero, so a non-zero remainder whose sign differs
 * from v's is moved by one v ("Why it is safe", the sign fix-up). */
int64_t oracle_floor_mod(int64_t x, int64_t v) {
    if (v == -1) return 0; /* INT64_MIN % -1 overflows in C; every x is a multiple of -1 */
    int64_t r = x % v;
    if (r != 0 && ((r < 0) != (v < 0))) r += v;
    return r;
}

static int64_t load_id(const void* p, int id_bytes, int64_t i) {
    if (id_bytes == 4) return (int64_t)((const int32_t*)p)[i];
    return ((const int64_t*)p)[i];
}

/* Per-token (request, offset) index, by a linear scan over cu_seqlens
 * ("What", second observation; "Why it is safe", the decode/prefill note:
 * a decode is one token per request at offset 0). */
int oracle_token_index(const int32_t* cu_seqlens, int32_t num_requests, int64_t num_tokens,
                       int is_decode, int32_t* req, int32_t* local) {
    if (num_tokens < 0 || num_requests < 0) return ORC_ERR_ARG;
    if (num_tokens == 0) return ORC_OK;
    if (!req || !local) return ORC_ERR_ARG;
    if (is_decode) {
        if ((int64_t)num_requests != num_tokens) return ORC_ERR_INDEX;
        for (int64_t t = 0; t < num_tokens; ++t) {
            req[t] = (int32_t)t;
            local[t] = 0;
        }
        return ORC_OK;
    }
    if (!cu_seqlens || num_requests < 1) return ORC_ERR_ARG;
    if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[num_requests] != num_tokens) return ORC_ERR_INDEX;
    /* the whole layout is checked before any write, so every token written
     * lies in [0, num_tokens) */
    for (int32_t r = 0; r < num_requests; ++r)
        if (cu_seqlens[r + 1] < cu_seqlens[r]) return ORC_ERR_INDEX;
    for (int32_t r = 0; r < num_requests; ++r) {
        for (int32_t t = cu_seqlens[r]; t < cu_seqlens[r + 1]; ++t) {
            req[t] = r;
            local[t] = t - cu_seqlens[r];
        }
    }
    return ORC_OK;
}

/* Checks that (req, local) describes B requests whose tokens sit contiguously
 * and in order in the flat batch, which is what packing ragged requests
 * produces.  Fills len[r]. */
static int check_index(const int32_t* req, const int32_t* local, int64_t T, int32_t B, int64_t* len,
                       int64_t* start) {
    for (int32_t r = 0; r < B; ++r) {
        len[r] = 0;
        start[r] = -1;
    }
    for (int64_t t = 0; t < T; ++t) {
        int32_t r = req[t];
        if (r < 0 || r >= B || local[t] < 0 || (int64_t)local[t] > t) return ORC_ERR_INDEX;
        int64_t s = t - (int64_t)local[t];
        if (start[r] < 0) start[r] = s;
        if (s != start[r] || (int64_t)local[t] != len[r]) return ORC_ERR_INDEX;
        len[r] += 1;
    }
    return ORC_OK;
}

static int row_ids_impl(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                        const int32_t* local, const void* ngram_context, int32_t B, int32_t ctx_len,
                        const int64_t* M, const int64_t* vocab, const int64_t* off, int32_t H,
                        int32_t N, int32_t hpn, int32_t L, int64_t b, int invalid_as_zero,
                        int64_t* out) {
    if (T < 0 || B < 0 || L < 1 || N < 2 || hpn < 1) return ORC_ERR_ARG;
    if (id_bytes != 4 && id_bytes != 8) return ORC_ERR_ARG;
    /* "Why it is safe", last point: the two geometry preconditions. */
    if (ctx_len != N - 1) return ORC_ERR_GEOMETRY;
    if ((int64_t)H != (int64_t)(N - 1) * hpn) return ORC_ERR_GEOMETRY;
    if (T == 0) return ORC_OK;
    if (!input_ids || !req || !local || !ngram_context || !M || !vocab || !off || !out || B < 1)
        return ORC_ERR_ARG;
    for (int64_t i = 0; i < (int64_t)L * H; ++i)
        if (vocab[i] == 0) return ORC_ERR_VOCAB;

    int rc = ORC_OK;
    int64_t* len = (int64_t*)malloc(sizeof(int64_t) * (size_t)B);
    int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)B);
    int64_t* W = NULL;
    int64_t* lastb = NULL;
    int64_t* V = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    if (!len || !start || !V) {
        rc = ORC_ERR_ALLOC;
        goto done;
    }
    rc = check_index(req, local, T, B, len, start);
    if (rc != ORC_OK) goto done;

    /* 1. Pack the window: an eos-filled [B, ctx + max_len] buffer, the
     *    context first (oldest id in column 0), then the request's tokens. */
    int64_t max_len = 0;
    for (int32_t r = 0; r < B; ++r)
        if (len[r] > max_len) max_len = len[r];
    const int64_t width = (int64_t)ctx_len + max_len;
    W = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B * width));
    lastb = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B * width));
    if (!W || !lastb) {
        rc = ORC_ERR_ALLOC;
        goto done;
    }
    for (int64_t i = 0; i < (int64_t)B * width; ++i) W[i] = b;
    for (int32_t r = 0; r < B; ++r)
        for (int32_t c = 0; c < ctx_len; ++c)
            W[(int64_t)r * width + c] = load_id(ngram_context, id_bytes, (int64_t)r * ctx_len + c);
    for (int64_t t = 0; t < T; ++t)
        W[(int64_t)req[t] * width + ctx_len + local[t]] = load_id(input_ids, id_bytes, t);

    /* 2. Boundary scan over the whole window, cummax style: lastb[r][q] is
     *    the largest q' <= q holding the boundary id, or -1. */
    for (int32_t r = 0; r < B; ++r) {
        int64_t run = -1;
        for (int64_t q = 0; q < width; ++q) {
            if (W[(int64_t)r * width + q] == b) run = q;
            lastb[(int64_t)r * width + q] = run;
        }
    }

    /* 3. Shifted values and the per-order hash for every real token. */
    for (int64_t t = 0; t < T; ++t) {
        const int64_t r = req[t];
        const int64_t p = (int64_t)ctx_len + local[t];
        const int64_t* row = W + r * width;
        for (int32_t s = 0; s < N; ++s) {
            /* valid iff p-s >= 0 and no boundary in [p-s, p-1]; for s = 0
             * the interval is empty. */
            int valid = (p - s >= 0) && (s == 0 || lastb[r * width + p - 1] < p - s);
            if (valid)
                V[s] = row[p - s];
            else
                V[s] = invalid_as_zero ? 0 : b;
        }
        for (int32_t l = 0; l < L; ++l) {
            for (int32_t n = 2; n <= N; ++n) {
                int64_t mix = 0;
                for (int32_t s = 0; s < n; ++s) mix ^= wrap_mul(V[s], M[(int64_t)l * N + s]);
                for (int32_t j = 0; j < hpn; ++j) {
                    const int64_t h = (int64_t)(n - 2) * hpn + j;
                    const int64_t k = (int64_t)l * H + h;
                    out[((int64_t)l * T + t) * H + h] = wrap_add(oracle_floor_mod(mix, vocab[k]), off[k]);
                }
            }
        }
    }

done:
    free(len);
    free(start);
    free(W);
    free(lastb);
    free(V);
    return rc;
}

/* The context each request carries into its next call: the last ctx_len ids
 * of (its ngram_context row, then its tokens of this batch), oldest first
 * ("What", second observation: ngram_context holds each request's ids just
 * before the batch).  A request with no token in the batch keeps its row.
 * (req, local) must describe a packed batch, as for oracle_row_ids. */
int oracle_next_context(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                        const int32_t* local, const void* ngram_context, int32_t B,
                        int32_t ctx_len, void* next_context) {
    if (T < 0 || B < 1 || ctx_len < 0 || (id_bytes != 4 && id_bytes != 8)) return ORC_ERR_ARG;
    if (!ngram_context || !next_context || (T > 0 && (!input_ids || !req || !local)))
        return ORC_ERR_ARG;
    int rc = ORC_OK;
    int64_t* len = (int64_t*)malloc(sizeof(int64_t) * (size_t)B);
    int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)B);
    int64_t* seq = NULL;
    if (!len || !start) {
        rc = ORC_ERR_ALLOC;
        goto done;
    }
    rc = check_index(req, local, T, B, len, start);
    if (rc != ORC_OK) goto done;
    for (int32_t r = 0; r < B; ++r) {
        /* the request's whole known history: context row, then its tokens */
        const int64_t n = (int64_t)ctx_len + len[r];
        free(seq);
        seq = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
        if (!seq) {
            rc = ORC_ERR_ALLOC;
            goto done;
        }
        for (int32_t c = 0; c < ctx_len; ++c)
            seq[c] = load_id(ngram_context, id_bytes, (int64_t)r * ctx_len + c);
        for (int64_t i = 0; i < len[r]; ++i) seq[ctx_len + i] = load_id(input_ids, id_bytes, start[r] + i);
        for (int32_t c = 0; c < ctx_len; ++c) {
            const int64_t v = seq[n - ctx_len + c];
            if (id_bytes == 4)
                ((int32_t*)next_context)[(int64_t)r * ctx_len + c] = (int32_t)v;
            else
                ((int64_t*)next_context)[(int64_t)r * ctx_len + c] = v;
        }
    }
done:
    free(len);
    free(start);
    free(seq);
    return rc;
}

/* bfloat16 bits to a double: the bits are the top half of an IEEE float. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The consumer of the row ids ("What": the ids are table row ids): for each
 * layer l and token t, the sum over heads of the table rows they name,
 *   emb[l][t][:] = sum_h table[l][row(l,t,h)][:],
 * with table [L, V, D] bfloat16 bits; a row id outside [0, V) adds nothing.
 * The sum is taken in double (exact for these inputs); abs_sum receives
 * sum_h |table[l][row][:]| for the floating-point error bound of a float
 * accumulation.  out and abs_sum are [L, T, D] doubles. */
int oracle_row_embed(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                     const int32_t* local, const void* ngram_context, int32_t B, int32_t ctx_len,
                     const int64_t* M, const int64_t* vocab, const int64_t* off, int32_t H,
                     int32_t N, int32_t hpn, int32_t L, int64_t b, const uint16_t* table,
                     int64_t V, int32_t D, double* out, double* abs_sum) {
    if (V < 0 || D < 1 || (T > 0 && (!table || !out || !abs_sum))) return ORC_ERR_ARG;
    if (T == 0) return ORC_OK;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L * T * H));
    if (!rows) return ORC_ERR_ALLOC;
    int rc = row_ids_impl(input_ids, id_bytes, T, req, local, ngram_context, B, ctx_len, M, vocab,
                          off, H, N, hpn, L, b, 0, rows);
    if (rc == ORC_OK) {
        for (int32_t l = 0; l < L; ++l) {
            for (int64_t t = 0; t < T; ++t) {
                double* o = out + ((int64_t)l * T + t) * D;
                double* a = abs_sum + ((int64_t)l * T + t) * D;
                for (int32_t d = 0; d < D; ++d) o[d] = a[d] = 0.0;
                for (int32_t h = 0; h < H; ++h) {
                    const int64_t row = rows[((int64_t)l * T + t) * H + h];
                    if (row < 0 || row >= V) continue;
                    const uint16_t* e = table + ((int64_t)l * V + row) * D;
                    for (int32_t d = 0; d < D; ++d) {
                        const double x = bf16_to_double(e[d]);
                        o[d] += x;
                        a[d] += x < 0 ? -x : x;
                    }
                }
            }
        }
    }
    free(rows);
    return rc;
}

/* Row ids under reading A (an invalid shift hashes the boundary id).
 * Arguments mean what they mean for the CUDA library's ple_row_ids; every
 * pointer is a host pointer.  out is [L, T, H] int64. */
int oracle_row_ids(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                   const int32_t* local, const void* ngram_context, int32_t B, int32_t ctx_len,
                   const int64_t* M, const int64_t* vocab, const int64_t* off, int32_t H, int32_t N,
                   int32_t hpn, int32_t L, int64_t b, int64_t* out) {
    return row_ids_impl(input_ids, id_bytes, T, req, local, ngram_context, B, ctx_len, M, vocab, off,
                        H, N, hpn, L, b, 0, out);
}

/* The same under reading B (an invalid shift contributes 0 to the XOR).
 * Kept only so the tests can show where the two readings part. */
int oracle_row_ids_reading_b(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                             const int32_t* local, const void* ngram_context, int32_t B,
                             int32_t ctx_len, const int64_t* M, const int64_t* vocab,
                             const int64_t* off, int32_t H, int32_t N, int32_t hpn, int32_t L,
                             int64_t b, int64_t* out) {
    return row_ids_impl(input_ids, id_bytes, T, req, local, ngram_context, B, ctx_len, M, vocab, off,
                        H, N, hpn, L, b, 1, out);
}
