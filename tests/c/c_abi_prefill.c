/*
 * A C program that drives the library through include/ple.h alone (no
 * Python), as a C caller would, and checks every result against the oracle
 * (oracle/ple_oracle.c, linked as test infrastructure).
 *
 * It builds a seeded ragged batch on the host (splitmix64: 37 requests,
 * some empty, ngram_size 4, 4 heads per order, 3 layers, 20 % boundary ids,
 * signed full-range multipliers, prime-ish vocab sizes), copies it to the
 * device, and runs:
 *   - ple_row_ids_ex in one launch (requests found from cu_seqlens) with the
 *     next call's context carried out;
 *   - ple_build_token_index followed by ple_row_ids;
 *   - ple_prepare_heads followed by ple_row_ids_ex with the prepared heads;
 *   - ple_row_ids_i32 (the low 32 bits of every row id);
 *   - a geometry the library refuses (ctx_len != ngram_size - 1), which must
 *     return PLE_ERR_GEOMETRY_CTX and leave the output untouched.
 * Exit status 0 when everything matches, 1 otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ple.h"

int oracle_token_index(const int32_t* cu_seqlens, int32_t num_requests, int64_t num_tokens,
                       int is_decode, int32_t* req, int32_t* local);
int oracle_row_ids(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                   const int32_t* local, const void* ngram_context, int32_t B, int32_t ctx_len,
                   const int64_t* M, const int64_t* vocab, const int64_t* off, int32_t H, int32_t N,
                   int32_t hpn, int32_t L, int64_t b, int64_t* out);
int oracle_next_context(const void* input_ids, int id_bytes, int64_t T, const int32_t* req,
                        const int32_t* local, const void* ngram_context, int32_t B,
                        int32_t ctx_len, void* out);

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64(void) { /* splitmix64 */
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

#define CHECK(call)                                                               \
    do {                                                                          \
        cudaError_t e_ = (call);                                                  \
        if (e_ != cudaSuccess) {                                                  \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));          \
            return 2;                                                             \
        }                                                                         \
    } while (0)

static int expect_status(const char* what, ple_status st, ple_status want) {
    if (st != want) {
        fprintf(stderr, "%s: status %d (%s), expected %d\n", what, (int)st,
                ple_status_string(st), (int)want);
        return 1;
    }
    return 0;
}

int main(void) {
    enum { B = 37, N = 4, HPN = 4, H = (N - 1) * HPN, L = 3, C = N - 1 };
    const int64_t boundary = 151643;
    int32_t cu[B + 1];
    cu[0] = 0;
    for (int r = 0; r < B; ++r) cu[r + 1] = cu[r] + (int32_t)(next_u64() % 200u) * (r % 7 != 3);
    const int64_t T = cu[B];
    int64_t* ids = malloc(sizeof(int64_t) * T);
    int64_t ctx[B * C], M[L * N], vocab[L * H], off[L * H];
    for (int64_t t = 0; t < T; ++t)
        ids[t] = (next_u64() % 5u == 0) ? boundary : (int64_t)(next_u64() % 151936u);
    for (int i = 0; i < B * C; ++i)
        ctx[i] = (next_u64() % 5u == 0) ? boundary : (int64_t)(next_u64() % 151936u);
    for (int i = 0; i < L * N; ++i) M[i] = (int64_t)next_u64();
    for (int l = 0; l < L; ++l) {
        int64_t acc = 0;
        for (int h = 0; h < H; ++h) {
            vocab[l * H + h] = (int64_t)(131071 + 2 * (next_u64() % 400000u));
            off[l * H + h] = acc;
            acc += vocab[l * H + h];
        }
    }

    /* the oracle's rows and carried context */
    int32_t* req = malloc(sizeof(int32_t) * T);
    int32_t* local = malloc(sizeof(int32_t) * T);
    int64_t* expect = malloc(sizeof(int64_t) * L * T * H);
    int64_t expect_ctx[B * C];
    if (oracle_token_index(cu, B, T, 0, req, local) ||
        oracle_row_ids(ids, 8, T, req, local, ctx, B, C, M, vocab, off, H, N, HPN, L, boundary,
                       expect) ||
        oracle_next_context(ids, 8, T, req, local, ctx, B, C, expect_ctx)) {
        fprintf(stderr, "oracle failed\n");
        return 2;
    }

    void *d_ids, *d_ctx, *d_M, *d_vocab, *d_off, *d_cu, *d_req, *d_local, *d_out, *d_out32,
        *d_next, *d_heads;
    CHECK(cudaMalloc(&d_ids, sizeof(int64_t) * T));
    CHECK(cudaMalloc(&d_ctx, sizeof ctx));
    CHECK(cudaMalloc(&d_M, sizeof M));
    CHECK(cudaMalloc(&d_vocab, sizeof vocab));
    CHECK(cudaMalloc(&d_off, sizeof off));
    CHECK(cudaMalloc(&d_cu, sizeof cu));
    CHECK(cudaMalloc(&d_req, sizeof(int32_t) * T));
    CHECK(cudaMalloc(&d_local, sizeof(int32_t) * T));
    CHECK(cudaMalloc(&d_out, sizeof(int64_t) * L * T * H));
    CHECK(cudaMalloc(&d_out32, sizeof(int32_t) * L * T * H));
    CHECK(cudaMalloc(&d_next, sizeof ctx));
    CHECK(cudaMalloc(&d_heads, (size_t)PLE_HEAD_BYTES * L * H));
    CHECK(cudaMemcpy(d_ids, ids, sizeof(int64_t) * T, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_ctx, ctx, sizeof ctx, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_M, M, sizeof M, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_vocab, vocab, sizeof vocab, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_off, off, sizeof off, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_cu, cu, sizeof cu, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CHECK(cudaStreamCreate(&stream));

    int64_t* got = malloc(sizeof(int64_t) * L * T * H);
    int32_t* got32 = malloc(sizeof(int32_t) * L * T * H);
    int64_t got_ctx[B * C];
    int bad = 0;

    /* one launch: requests from cu_seqlens, context carried */
    bad |= expect_status("ple_row_ids_ex (one launch)",
                         ple_row_ids_ex(d_ids, PLE_I64, T, NULL, NULL, d_ctx, B, C, d_M, d_vocab,
                                        d_off, H, N, HPN, L, boundary, d_out, PLE_I64, d_cu,
                                        d_next, NULL, stream),
                         PLE_OK);
    CHECK(cudaStreamSynchronize(stream));
    CHECK(cudaMemcpy(got, d_out, sizeof(int64_t) * L * T * H, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(got_ctx, d_next, sizeof ctx, cudaMemcpyDeviceToHost));
    if (memcmp(got, expect, sizeof(int64_t) * L * T * H)) bad |= 1, fprintf(stderr, "one-launch rows differ\n");
    if (memcmp(got_ctx, expect_ctx, sizeof ctx)) bad |= 1, fprintf(stderr, "carried context differs\n");

    /* the page's two steps: index, then the hash reading it */
    CHECK(cudaMemset(d_out, 0, sizeof(int64_t) * L * T * H));
    bad |= expect_status("ple_build_token_index",
                         ple_build_token_index(d_cu, B, T, 0, d_req, d_local, stream), PLE_OK);
    bad |= expect_status("ple_row_ids",
                         ple_row_ids(d_ids, PLE_I64, T, d_req, d_local, d_ctx, B, C, d_M, d_vocab,
                                     d_off, H, N, HPN, L, boundary, d_out, stream),
                         PLE_OK);
    CHECK(cudaStreamSynchronize(stream));
    CHECK(cudaMemcpy(got, d_out, sizeof(int64_t) * L * T * H, cudaMemcpyDeviceToHost));
    if (memcmp(got, expect, sizeof(int64_t) * L * T * H)) bad |= 1, fprintf(stderr, "indexed rows differ\n");

    /* prepared head constants */
    CHECK(cudaMemset(d_out, 0, sizeof(int64_t) * L * T * H));
    bad |= expect_status("ple_prepare_heads",
                         ple_prepare_heads(d_vocab, d_off, L, H, d_heads, stream), PLE_OK);
    bad |= expect_status("ple_row_ids_ex (prepared)",
                         ple_row_ids_ex(d_ids, PLE_I64, T, NULL, NULL, d_ctx, B, C, d_M, NULL, NULL,
                                        H, N, HPN, L, boundary, d_out, PLE_I64, d_cu, NULL, d_heads,
                                        stream),
                         PLE_OK);
    CHECK(cudaStreamSynchronize(stream));
    CHECK(cudaMemcpy(got, d_out, sizeof(int64_t) * L * T * H, cudaMemcpyDeviceToHost));
    if (memcmp(got, expect, sizeof(int64_t) * L * T * H)) bad |= 1, fprintf(stderr, "prepared rows differ\n");

    /* int32 row ids: the low 32 bits */
    bad |= expect_status("ple_row_ids_i32",
                         ple_row_ids_i32(d_ids, PLE_I64, T, d_req, d_local, d_ctx, B, C, d_M,
                                         d_vocab, d_off, H, N, HPN, L, boundary,
                                         (int32_t*)d_out32, stream),
                         PLE_OK);
    CHECK(cudaStreamSynchronize(stream));
    CHECK(cudaMemcpy(got32, d_out32, sizeof(int32_t) * L * T * H, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < (int64_t)L * T * H; ++i)
        if (got32[i] != (int32_t)(uint32_t)(uint64_t)expect[i]) {
            bad |= 1;
            fprintf(stderr, "int32 row %lld differs\n", (long long)i);
            break;
        }

    /* a geometry the library refuses: nothing launched, output untouched */
    CHECK(cudaMemset(d_out, 0x5A, sizeof(int64_t) * L * T * H));
    bad |= expect_status("ple_row_ids (ctx_len wrong)",
                         ple_row_ids(d_ids, PLE_I64, T, d_req, d_local, d_ctx, B, C + 1, d_M,
                                     d_vocab, d_off, H, N, HPN, L, boundary, d_out, stream),
                         PLE_ERR_GEOMETRY_CTX);
    CHECK(cudaStreamSynchronize(stream));
    CHECK(cudaMemcpy(got, d_out, sizeof(int64_t) * L * T * H, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < (int64_t)L * T * H; ++i)
        if (got[i] != (int64_t)0x5A5A5A5A5A5A5A5Aull) {
            bad |= 1;
            fprintf(stderr, "output touched after a refused call\n");
            break;
        }

    printf("%s: T=%lld, B=%d, L=%d, H=%d\n", bad ? "MISMATCH" : "OK", (long long)T, B, L, H);
    return bad ? 1 : 0;
}
