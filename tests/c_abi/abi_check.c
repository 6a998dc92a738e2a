/*
 * Drives libhsi from plain C11 through include/hsi.h: the header compiles as C,
 * every call links, and the calls behave as documented.
 *
 *   abi_check host   -- no device needed: status strings, workspace sizes and
 *                       host-side argument checks (nothing is launched).
 *   abi_check gpu    -- one hsi_topk on device buffers, checked against the
 *                       top-k this file works out by hand, plus the sticky
 *                       device error word.
 *
 * Prints one line per failed check and exits with the number of failures.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "hsi.h"

static int failures = 0;

#define CHECK(cond)                                                          \
    do {                                                                     \
        if (!(cond)) {                                                       \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            ++failures;                                                      \
        }                                                                    \
    } while (0)

static int host_checks(void) {
    CHECK(strcmp(hsi_status_string(HSI_OK), "unknown status") != 0);
    CHECK(strcmp(hsi_status_string(HSI_ERR_TOO_LARGE), "unknown status") != 0);
    CHECK(strcmp(hsi_status_string(12345), "unknown status") == 0);

    /* short rows select in shared memory; long rows need scratch */
    CHECK(hsi_workspace_size(HSI_WS_TOPK, 4, 16384, 512) == 0);
    CHECK(hsi_workspace_size(HSI_WS_TOPK, 4, 1 << 20, 512) > 0);
    CHECK(hsi_workspace_size(HSI_WS_SCORE, 64, 1 << 20, 0) == 0);

    /* argument checks run before anything touches the device: these pointers
       are never dereferenced */
    const float* fs = (const float*)(uintptr_t)(1u << 20);
    const int32_t* fi = (const int32_t*)(uintptr_t)(1u << 20);
    int32_t* oi = (int32_t*)(uintptr_t)(1u << 20);
    float* ov = (float*)(uintptr_t)(1u << 20);
    CHECK(hsi_topk(NULL, 100, fi, 1, 100, 8, NULL, 0, 0, oi, ov, NULL, 0, NULL) == HSI_ERR_INVALID_ARG);
    CHECK(hsi_topk(fs, 100, fi, 1, 100, 0, NULL, 0, 0, oi, ov, NULL, 0, NULL) == HSI_ERR_INVALID_ARG);
    CHECK(hsi_topk(fs, 99, fi, 1, 100, 8, NULL, 0, 0, oi, ov, NULL, 0, NULL) == HSI_ERR_INVALID_ARG);
    CHECK(hsi_topk(fs, 1 << 20, fi, 4, 1 << 20, 512, NULL, 0, 0, oi, ov, NULL, 0, NULL) == HSI_ERR_WORKSPACE);
    CHECK(hsi_topk_noalloc(fs, 1 << 20, fi, 57, 1 << 20, 512, NULL, 0, 0, oi, ov, NULL) == HSI_ERR_TOO_LARGE);
    return failures;
}

/* Scores of row b at position i: a permutation of 0..n-1 scaled by (b + 1),
   so the top-k of a row of length n are the positions holding n-1, n-2, ... */
#define N_ROW 5003   /* prime: i -> (i * 7919) mod N_ROW is a permutation */
#define B_ROWS 3
#define K_SEL 64

static float score_at(int b, int i) { return (float)((int64_t)i * 7919 % N_ROW) * (float)(b + 1); }

static int gpu_checks(void) {
    static float h_scores[B_ROWS * N_ROW];
    int32_t h_n[B_ROWS] = {N_ROW, N_ROW - 1000, 10};
    for (int b = 0; b < B_ROWS; ++b)
        for (int i = 0; i < N_ROW; ++i) h_scores[b * N_ROW + i] = score_at(b, i);

    float *d_scores = NULL, *d_val = NULL;
    int32_t *d_n = NULL, *d_idx = NULL;
    void* ws = NULL;
    size_t ws_bytes = hsi_workspace_size(HSI_WS_TOPK, B_ROWS, N_ROW, K_SEL);
    if (cudaMalloc((void**)&d_scores, sizeof h_scores) != cudaSuccess ||
        cudaMalloc((void**)&d_n, sizeof h_n) != cudaSuccess ||
        cudaMalloc((void**)&d_idx, B_ROWS * K_SEL * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc((void**)&d_val, B_ROWS * K_SEL * sizeof(float)) != cudaSuccess ||
        (ws_bytes && cudaMalloc(&ws, ws_bytes) != cudaSuccess)) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    CHECK(hsi_device_check() == HSI_OK);
    cudaMemcpy(d_scores, h_scores, sizeof h_scores, cudaMemcpyHostToDevice);
    cudaMemcpy(d_n, h_n, sizeof h_n, cudaMemcpyHostToDevice);
    CHECK(hsi_topk(d_scores, N_ROW, d_n, B_ROWS, N_ROW, K_SEL, NULL, 0, 0, d_idx, d_val, ws, ws_bytes, NULL) ==
          HSI_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(hsi_device_error(NULL) == HSI_OK);

    int32_t h_idx[B_ROWS * K_SEL];
    float h_val[B_ROWS * K_SEL];
    cudaMemcpy(h_idx, d_idx, sizeof h_idx, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_val, d_val, sizeof h_val, cudaMemcpyDeviceToHost);
    for (int b = 0; b < B_ROWS; ++b) {
        /* expected: the visible positions in descending score order (scores are
           distinct within a row), then -1 / -inf past the row's length */
        int taken = 0;
        int32_t want_idx[K_SEL];
        float last = 1e30f;
        for (int r = 0; r < K_SEL; ++r) want_idx[r] = -1;
        for (int r = 0; r < K_SEL && r < h_n[b]; ++r) {
            int best = -1;
            for (int i = 0; i < h_n[b]; ++i) {
                float s = score_at(b, i);
                if (s < last && (best < 0 || s > score_at(b, best))) best = i;
            }
            want_idx[r] = best;
            last = score_at(b, best);
            ++taken;
        }
        for (int r = 0; r < K_SEL; ++r) {
            CHECK(h_idx[b * K_SEL + r] == want_idx[r]);
            if (r < taken) CHECK(h_val[b * K_SEL + r] == score_at(b, want_idx[r]));
            else CHECK(h_val[b * K_SEL + r] < -1e38f);
        }
    }
    cudaFree(d_scores);
    cudaFree(d_n);
    cudaFree(d_idx);
    cudaFree(d_val);
    if (ws) cudaFree(ws);
    return failures;
}

int main(int argc, char** argv) {
    if (argc != 2 || (strcmp(argv[1], "host") && strcmp(argv[1], "gpu"))) {
        fprintf(stderr, "usage: %s host|gpu\n", argv[0]);
        return 2;
    }
    int f = strcmp(argv[1], "host") == 0 ? host_checks() : gpu_checks();
    printf("%s: %d failure(s)\n", argv[1], f);
    return f;
}
