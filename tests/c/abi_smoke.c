/*
 * abi_smoke.c -- the C ABI used from plain C (C11, no C++): include/kda.h compiles on its
 * own, and a small prefill runs through kda_chunk_fwd (device buffers) and
 * kda_chunk_fwd_host (host buffers, streamed), which must agree bit for bit; argument
 * errors come back as status codes.  Built and run by tests/test_c_abi.py.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"

#define CHECK(x)                                                               \
    do {                                                                       \
        if (!(x)) {                                                            \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #x);  \
            return 1;                                                          \
        }                                                                      \
    } while (0)

/* xorshift64*: a deterministic source of inputs (no attention arithmetic here) */
static uint64_t rng_state = 0x4B4441ull;
static float urand(void) {
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (float)((rng_state * 2685821657736338717ull) >> 40) / (float)(1u << 24);
}

int main(void) {
    const int B = 1, H = 2, D = 128;
    const int64_t T = 300;
    const size_t tok = (size_t)B * T * H; /* token-heads */
    float* q = malloc(tok * D * 4);
    float* k = malloc(tok * D * 4);
    float* v = malloc(tok * D * 4);
    float* la = malloc(tok * D * 4);
    float* beta = malloc(tok * 4);
    float* out_a = malloc(tok * D * 4);
    float* out_b = malloc(tok * D * 4);
    float* fin_a = malloc((size_t)B * H * D * D * 4);
    float* fin_b = malloc((size_t)B * H * D * D * 4);
    CHECK(q && k && v && la && beta && out_a && out_b && fin_a && fin_b);
    for (size_t r = 0; r < tok; ++r) {
        float nq = 0.f, nk = 0.f;
        for (int c = 0; c < D; ++c) {
            q[r * D + c] = urand() - 0.5f;
            k[r * D + c] = urand() - 0.5f;
            v[r * D + c] = 2.f * urand() - 1.f;
            la[r * D + c] = -0.001f - 0.099f * urand();
            nq += q[r * D + c] * q[r * D + c];
            nk += k[r * D + c] * k[r * D + c];
        }
        for (int c = 0; c < D; ++c) { /* unit rows, as the caller's normalisation */
            q[r * D + c] /= sqrtf(nq);
            k[r * D + c] /= sqrtf(nk);
        }
        beta[r] = 0.25f + 0.5f * urand();
    }

    /* device call */
    void *dq, *dk, *dv, *dla, *dbeta, *dout;
    float* dfin;
    CHECK(cudaMalloc(&dq, tok * D * 4) == cudaSuccess && cudaMalloc(&dk, tok * D * 4) == cudaSuccess &&
          cudaMalloc(&dv, tok * D * 4) == cudaSuccess && cudaMalloc(&dla, tok * D * 4) == cudaSuccess &&
          cudaMalloc(&dbeta, tok * 4) == cudaSuccess && cudaMalloc(&dout, tok * D * 4) == cudaSuccess &&
          cudaMalloc((void**)&dfin, (size_t)B * H * D * D * 4) == cudaSuccess);
    CHECK(cudaMemcpy(dq, q, tok * D * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dk, k, tok * D * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dv, v, tok * D * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dla, la, tok * D * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dbeta, beta, tok * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    /* one int per (sequence, head), rounded up to 256 bytes, then 256 bytes of unit counters */
    const size_t cws_bytes = kda_workspace_size(KDA_OP_CHUNK, B, T, H, D, D, 64);
    CHECK(cws_bytes == (((size_t)B * H * 4 + 255) / 256) * 256 + 256);
    void* cws;
    CHECK(cudaMalloc(&cws, cws_bytes) == cudaSuccess);
    CHECK(kda_chunk_fwd(dq, dk, dv, dla, dbeta, NULL, dout, dfin, B, T, H, D, D, 64, KDA_F32, KDA_F32, NULL, 0,
                        NULL) == KDA_ERR_WORKSPACE);
    CHECK(kda_chunk_fwd(dq, dk, dv, dla, dbeta, NULL, dout, dfin, B, T, H, D, D, 64, KDA_F32, KDA_F32, cws,
                        cws_bytes, NULL) == KDA_OK);
    CHECK(cudaMemcpy(out_a, dout, tok * D * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(fin_a, dfin, (size_t)B * H * D * D * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(kda_get_device_status(NULL) == KDA_OK);

    /* host-buffer call, 128-token segments */
    size_t ws_bytes = kda_host_fwd_workspace_size(B, H, D, D, 128, KDA_F32, KDA_F32);
    void* ws;
    CHECK(ws_bytes > 0 && cudaMalloc(&ws, ws_bytes) == cudaSuccess);
    CHECK(kda_chunk_fwd_host(q, k, v, la, beta, NULL, out_b, fin_b, B, T, H, D, D, KDA_F32, KDA_F32, 128, ws,
                             ws_bytes, NULL) == KDA_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(memcmp(out_a, out_b, tok * D * 4) == 0);
    CHECK(memcmp(fin_a, fin_b, (size_t)B * H * D * D * 4) == 0);

    /* argument errors are status codes */
    CHECK(kda_chunk_fwd(dq, dk, dv, dla, dbeta, NULL, dout, dfin, B, T, H, 64, D, 64, KDA_F32, KDA_F32, cws,
                        cws_bytes, NULL) == KDA_ERR_UNSUPPORTED);
    CHECK(kda_chunk_fwd(NULL, dk, dv, dla, dbeta, NULL, dout, dfin, B, T, H, D, D, 64, KDA_F32, KDA_F32, cws,
                        cws_bytes, NULL) == KDA_ERR_INVALID_ARG);
    CHECK(strncmp(kda_status_string(KDA_ERR_MISALIGNED), "KDA_", 4) == 0);
    printf("abi_smoke ok\n");
    return 0;
}
