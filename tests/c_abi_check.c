/*
 * A plain C caller of libpgt.so: include/pgt.h plus the CUDA runtime, nothing else.
 *
 *   c_abi_check cpu   argument checks that need no GPU (exit 0 when all statuses match)
 *   c_abi_check gpu   preamble, an all-ones GEMM (every element must equal K exactly, in
 *                     every scheduler mode), bit-identical outputs across modes on
 *                     pseudo-random data (also striped work stealing through the
 *                     descriptor form), the add, pgt_last_error, destroy
 */
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pgt.h"

static int failures = 0;

static void expect(const char* what, int got, int want) {
    if (got != want) {
        printf("FAIL %s: got %d (%s), want %d\n", what, got, pgt_strerror(got), want);
        ++failures;
    }
}

static uint16_t bf16_of(float f) { /* round to nearest even; finite inputs only */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

static int cpu_checks(void) {
    /* the descriptor layout the C compiler uses, for the binding to compare with its own */
    printf("layout pgt_gemm_desc %zu dtype %zu ws_groups %zu epilogue %zu alpha %zu ws_layout %zu bias %zu\n",
           sizeof(pgt_gemm_desc), offsetof(pgt_gemm_desc, dtype), offsetof(pgt_gemm_desc, ws_groups),
           offsetof(pgt_gemm_desc, epilogue), offsetof(pgt_gemm_desc, alpha), offsetof(pgt_gemm_desc, ws_layout),
           offsetof(pgt_gemm_desc, bias));
    printf("layout pgt_gemm_plan_info %zu pgt_trace %zu pgt_scale_space %zu\n", sizeof(pgt_gemm_plan_info),
           sizeof(pgt_trace), sizeof(pgt_scale_space));
    pgt_ctx* ctx = (pgt_ctx*)0x1;
    expect("preamble null out", pgt_preamble(0, 8, 0, NULL), PGT_ERR_ARG);
    expect("preamble groups 0", pgt_preamble(0, 0, 0, &ctx), PGT_ERR_ARG);
    if (ctx != NULL) { printf("FAIL preamble did not clear *out\n"); ++failures; }
    expect("num_sms null", pgt_num_sms(NULL), PGT_ERR_ARG);
    expect("destroy null", pgt_destroy(NULL), PGT_OK);
    expect("plan null", pgt_gemm_plan(NULL, NULL, NULL), PGT_ERR_ARG);
    if (pgt_gemm_workspace_bytes(NULL) != 0) { printf("FAIL workspace null\n"); ++failures; }
    pgt_gemm_desc d;
    memset(&d, 0, sizeof(d));
    d.M = 8192; d.N = 8192; d.K = 8192; d.dtype = PGT_MXFP8; d.b_layout = PGT_B_NK;
    if (pgt_gemm_workspace_bytes(&d) != 2u * 16u * 64u * 512u) { printf("FAIL mxfp8 workspace size\n"); ++failures; }
    if (strcmp(pgt_strerror(PGT_ERR_TIMEOUT), "device wait timed out") != 0) { printf("FAIL strerror\n"); ++failures; }
    /* the flat form checks its counter-group count before anything else */
    expect("flat ws_groups 65", pgt_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 64, 64, 64, PGT_BF16, PGT_B_KN,
                                         PGT_WORK_STEALING, 16, 65, NULL, 0, NULL), PGT_ERR_GROUPS);
    expect("flat ws_groups -1", pgt_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 64, 64, 64, PGT_BF16, PGT_B_KN,
                                         PGT_WORK_STEALING, 16, -1, NULL, 0, NULL), PGT_ERR_GROUPS);
    expect("flat null context", pgt_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 64, 64, 64, PGT_BF16, PGT_B_KN,
                                         PGT_WORK_STEALING, 16, 8, NULL, 0, NULL), PGT_ERR_ARG);
    return failures;
}

static int gpu_checks(void) {
    pgt_ctx* ctx = NULL;
    expect("preamble", pgt_preamble(0, 8, 0, &ctx), PGT_OK);
    if (ctx == NULL) return ++failures;
    const int M = 1000, N = 1104, K = 256;
    uint16_t* hA = (uint16_t*)malloc(sizeof(uint16_t) * M * K);
    uint16_t* hB = (uint16_t*)malloc(sizeof(uint16_t) * K * N);
    uint16_t* hC = (uint16_t*)malloc(sizeof(uint16_t) * M * N);
    uint16_t* hR = (uint16_t*)malloc(sizeof(uint16_t) * M * N);
    void *dA, *dB, *dC;
    cudaMalloc(&dA, sizeof(uint16_t) * M * K);
    cudaMalloc(&dB, sizeof(uint16_t) * K * N);
    cudaMalloc(&dC, sizeof(uint16_t) * M * N);
    const int modes[6] = {PGT_BLOCKED, PGT_INTERLEAVED, PGT_SWIZZLED, PGT_WORK_STEALING, PGT_BLOCKED_GROUPED_M,
                          PGT_LAUNCH_CONTROL};
    /* all ones: C = K exactly */
    for (int i = 0; i < M * K; ++i) hA[i] = bf16_of(1.0f);
    for (int i = 0; i < K * N; ++i) hB[i] = bf16_of(1.0f);
    cudaMemcpy(dA, hA, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, hB, sizeof(uint16_t) * K * N, cudaMemcpyHostToDevice);
    for (int m = 0; m < 6; ++m) {
        cudaMemset(dC, 0xFF, sizeof(uint16_t) * M * N);
        expect("gemm ones", pgt_gemm(ctx, dA, dB, NULL, NULL, dC, M, N, K, PGT_BF16, PGT_B_KN, modes[m], 4, 0, NULL,
                                     0, NULL), PGT_OK);
        cudaMemcpy(hC, dC, sizeof(uint16_t) * M * N, cudaMemcpyDeviceToHost);
        int bad = 0;
        for (int i = 0; i < M * N; ++i) bad += hC[i] != bf16_of((float)K);
        if (bad) { printf("FAIL all-ones mode %d: %d wrong elements\n", modes[m], bad); ++failures; }
    }
    /* pseudo-random small integers / 16 (exact in bf16): every mode gives the same bits */
    uint32_t s = 12345u;
    for (int i = 0; i < M * K; ++i) { s = s * 1664525u + 1013904223u; hA[i] = bf16_of((float)((int)(s >> 28) - 8) / 16.0f); }
    for (int i = 0; i < K * N; ++i) { s = s * 1664525u + 1013904223u; hB[i] = bf16_of((float)((int)(s >> 28) - 8) / 16.0f); }
    cudaMemcpy(dA, hA, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, hB, sizeof(uint16_t) * K * N, cudaMemcpyHostToDevice);
    for (int m = 0; m < 6; ++m) {
        expect("gemm random", pgt_gemm(ctx, dA, dB, NULL, NULL, dC, M, N, K, PGT_BF16, PGT_B_KN, modes[m], 16,
                                       m == 3 ? 3 : 0, NULL, 0, NULL), PGT_OK);
        cudaMemcpy(m == 0 ? hR : hC, dC, sizeof(uint16_t) * M * N, cudaMemcpyDeviceToHost);
        if (m > 0 && memcmp(hR, hC, sizeof(uint16_t) * M * N) != 0) {
            printf("FAIL mode %d differs from blocked\n", modes[m]);
            ++failures;
        }
    }
    /* the descriptor form: work stealing with striped tile ownership, same bits */
    {
        pgt_gemm_desc dd;
        memset(&dd, 0, sizeof(dd));
        dd.M = M; dd.N = N; dd.K = K; dd.dtype = PGT_BF16; dd.b_layout = PGT_B_KN;
        dd.sched_mode = PGT_WORK_STEALING; dd.group_size = 16; dd.ws_groups = 4; dd.ws_layout = PGT_WS_STRIPED;
        expect("gemm_ex striped", pgt_gemm_ex(ctx, &dd, dA, dB, NULL, NULL, dC, NULL, 0, NULL, NULL), PGT_OK);
        cudaMemcpy(hC, dC, sizeof(uint16_t) * M * N, cudaMemcpyDeviceToHost);
        if (memcmp(hR, hC, sizeof(uint16_t) * M * N) != 0) { printf("FAIL striped work stealing differs\n"); ++failures; }
        dd.ws_layout = 7;
        expect("gemm_ex bad layout", pgt_gemm_ex(ctx, &dd, dA, dB, NULL, NULL, dC, NULL, 0, NULL, NULL), PGT_ERR_ARG);
    }
    /* entries against a direct sum: every product is a multiple of 2^-8 below 2^-2 in size and
     * |sum| <= 64, so each fp32 partial sum is exact and C is that sum rounded once to bf16 */
    for (int t = 0; t < 64; ++t) {
        const int i = (t * 977) % M, j = (t * 331) % N;
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) {
            uint32_t ua = (uint32_t)hA[i * K + k] << 16, ub = (uint32_t)hB[k * N + j] << 16;
            float a, b;
            memcpy(&a, &ua, 4);
            memcpy(&b, &ub, 4);
            acc += a * b;
        }
        if (hR[i * N + j] != bf16_of(acc)) {
            printf("FAIL entry (%d,%d)\n", i, j);
            ++failures;
        }
    }
    /* the add */
    float *x, *y, *o;
    const int R = 300, Cc = 500;
    cudaMalloc((void**)&x, sizeof(float) * R * Cc);
    cudaMalloc((void**)&y, sizeof(float) * R * Cc);
    cudaMalloc((void**)&o, sizeof(float) * R * Cc);
    float* hx = (float*)malloc(sizeof(float) * R * Cc);
    for (int i = 0; i < R * Cc; ++i) hx[i] = (float)i * 0.5f;
    cudaMemcpy(x, hx, sizeof(float) * R * Cc, cudaMemcpyHostToDevice);
    cudaMemcpy(y, hx, sizeof(float) * R * Cc, cudaMemcpyHostToDevice);
    expect("add", pgt_add(ctx, x, y, o, R, Cc, 0, 0, 0, PGT_INTERLEAVED, 32, 16, 0, NULL, NULL), PGT_OK);
    cudaMemcpy(hx, o, sizeof(float) * R * Cc, cudaMemcpyDeviceToHost);
    for (int i = 0; i < R * Cc; ++i)
        if (hx[i] != (float)i) { printf("FAIL add at %d\n", i); ++failures; break; }
    int32_t detail[4];
    expect("last_error", pgt_last_error(ctx, NULL, detail), PGT_OK);
    expect("flat ws_groups above max_groups", pgt_gemm(ctx, dA, dB, NULL, NULL, dC, M, N, K, PGT_BF16, PGT_B_KN,
                                                       PGT_WORK_STEALING, 16, 9, NULL, 0, NULL), PGT_ERR_GROUPS);
    expect("bad ws_groups", pgt_gemm_plan(ctx, &(pgt_gemm_desc){.M = 64, .N = 64, .K = 64, .group_size = 1,
                                                                   .ws_groups = 9}, &(pgt_gemm_plan_info){0}),
           PGT_ERR_GROUPS);
    cudaFree(dA); cudaFree(dB); cudaFree(dC); cudaFree(x); cudaFree(y); cudaFree(o);
    free(hA); free(hB); free(hC); free(hR); free(hx);
    expect("destroy", pgt_destroy(ctx), PGT_OK);
    return failures;
}

int main(int argc, char** argv) {
    const int gpu = argc > 1 && strcmp(argv[1], "gpu") == 0;
    const int rc = gpu ? gpu_checks() : cpu_checks();
    printf("%s checks: %s\n", gpu ? "gpu" : "cpu", rc ? "FAILED" : "ok");
    return rc ? 1 : 0;
}
