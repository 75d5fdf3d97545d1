/*
 * The C ABI used from plain C, with no Python or PyTorch in the process: a
 * caller that owns its device memory through the CUDA runtime (cudaMalloc),
 * runs route -> dispatch -> synthetic expert -> combine through include/moe.h
 * for a bf16 and an fp8 batch, and the allocation-free route, then checks
 * every result against the CPU oracle (oracle/moe_oracle.c, linked into this
 * test program only; the library never sees it).
 *
 * Bars as in the GPU parity tests: indices, counts, offsets, slots and the
 * kept dispatched rows (bf16 bits, e4m3 codes, fp32 scales, recv_src) equal;
 * routing weights within 1e-6 relative; combine within 1 bf16 ulp.
 *
 * Build (the GPU test does this): gcc -O2 -std=c11 c_abi_check.c moe_oracle.c
 *   -I include -I <cuda>/include -L <lib dir> -lmoe_gb300 -L <cuda>/lib64
 *   -lcudart -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe.h"

/* the oracle's entry points (test infrastructure) */
int oracle_route(int32_t T, int32_t E, int32_t k, const float *logits, int32_t *topk_idx, float *topk_w,
                 double *topk_w64);
int oracle_count(int32_t T, int32_t E, int32_t k, int32_t R, int32_t C, const int32_t *topk_idx, int32_t *counts,
                 int32_t *offsets, int32_t *slot, int32_t *rank_counts, int32_t *dropped);
int oracle_dispatch_bf16(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C, const uint16_t *x,
                         const int32_t *topk_idx, const int32_t *slot, uint16_t *recv_x, int32_t *recv_src);
int oracle_dispatch_fp8(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C, const uint16_t *x,
                        const int32_t *topk_idx, const int32_t *slot, uint8_t *recv_q, float *recv_scale,
                        int32_t *recv_src);
int oracle_expert_synthetic(int32_t H, int32_t E, int32_t C, int32_t fp8, const void *recv, const float *recv_scale,
                            const int32_t *counts, const float *s, uint16_t *y);
int oracle_combine(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C, const uint16_t *y,
                   const int32_t *topk_idx, const float *topk_w, const int32_t *slot, uint16_t *out);

static int failures = 0;
#define CHECK(cond, ...)                                    \
    do {                                                    \
        if (!(cond)) {                                      \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                   \
            fprintf(stderr, "\n");                          \
            ++failures;                                     \
        }                                                   \
    } while (0)
#define CUDA(call)                                                                 \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
            exit(2);                                                               \
        }                                                                          \
    } while (0)
#define MOE(call)                                                                  \
    do {                                                                           \
        int r_ = (call);                                                           \
        if (r_ != MOE_OK) {                                                        \
            fprintf(stderr, "%s at %s:%d\n", moe_status_string(r_), __FILE__, __LINE__); \
            exit(3);                                                               \
        }                                                                          \
    } while (0)

/* A 64-bit LCG and Box-Muller: inputs only (no arithmetic of the method). */
static uint64_t rng_state;
static double uniform01(void) {
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    return ((rng_state >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}
static double normal(void) {
    const double u = uniform01(), v = uniform01();
    return sqrt(-2.0 * log(u)) * cos(6.283185307179586 * v);
}
/* bf16 bits of a float by truncation of a value that is a bf16 already (the
   inputs are drawn as bf16: a normal sample with its low 16 bits cleared) */
static uint16_t bf16_bits_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}
static int32_t ordered(uint16_t b) { return (b & 0x8000) ? 0x8000 - (b & 0x7FFF) : 0x8000 + (b & 0x7FFF); }

static void *dev_alloc(size_t bytes) {
    void *p = NULL;
    CUDA(cudaMalloc(&p, bytes > 0 ? bytes : 16));
    return p;
}

static void run_case(int32_t T, int32_t H, int32_t E, int32_t k, int32_t R, int32_t C, int fp8, uint64_t seed) {
    moe_problem p;
    memset(&p, 0, sizeof p);
    p.num_tokens = T; p.hidden = H; p.num_experts = E; p.top_k = k; p.num_ranks = R; p.capacity = C;
    p.dispatch_dtype = fp8 ? MOE_DTYPE_FP8_E4M3_B128 : MOE_DTYPE_BF16;
    CHECK(moe_validate(&p) == MOE_OK, "problem rejected");
    const size_t TH = (size_t)T * H, TK = (size_t)T * k, ECH = (size_t)E * C * H, EC = (size_t)E * C;
    const int32_t nb = H / 128;

    /* host inputs */
    rng_state = seed;
    uint16_t *x = malloc(TH * 2);
    float *logits = malloc((size_t)T * E * 4), *s = malloc((size_t)E * 4);
    for (size_t i = 0; i < TH; ++i) {
        float f = (float)normal();
        uint32_t u;
        memcpy(&u, &f, 4);
        u &= 0xFFFF0000u;
        memcpy(&f, &u, 4);
        x[i] = bf16_bits_of(f);
    }
    for (size_t i = 0; i < (size_t)T * E; ++i) logits[i] = (float)normal();
    for (int32_t e = 0; e < E; ++e) s[e] = 1.0f + (float)e / (float)E;

    /* device buffers, owned by this caller */
    void *d_x = dev_alloc(TH * 2), *d_recv = dev_alloc(ECH * (fp8 ? 1 : 2)), *d_y = dev_alloc(ECH * 2),
         *d_out = dev_alloc(TH * 2);
    float *d_logits = dev_alloc((size_t)T * E * 4), *d_w = dev_alloc(TK * 4), *d_s = dev_alloc((size_t)E * 4);
    float *d_scale = fp8 ? dev_alloc(EC * nb * 4) : NULL;
    int32_t *d_idx = dev_alloc(TK * 4), *d_slot = dev_alloc(TK * 4), *d_counts = dev_alloc((size_t)E * 4),
            *d_offsets = dev_alloc((size_t)(E + 1) * 4), *d_rank = dev_alloc((size_t)R * 4), *d_drop = dev_alloc(4),
            *d_src = dev_alloc(EC * 4);
    const size_t ws_bytes = moe_route_workspace_bytes(&p);
    void *d_ws = dev_alloc(ws_bytes);
    CUDA(cudaMemcpy(d_x, x, TH * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_logits, logits, (size_t)T * E * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_s, s, (size_t)E * 4, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CUDA(cudaStreamCreate(&st));
    MOE(moe_route(&p, d_logits, d_idx, d_w, d_counts, d_offsets, d_slot, d_rank, d_drop, d_ws, ws_bytes, st));
    MOE(moe_dispatch(&p, d_x, d_idx, d_slot, d_recv, d_scale, d_src, st));
    MOE(moe_expert_synthetic(&p, d_recv, d_scale, d_counts, d_s, d_y, st));
    MOE(moe_combine(&p, d_y, d_idx, d_w, d_slot, d_out, st));
    CUDA(cudaStreamSynchronize(st));
    CHECK(moe_device_status() == MOE_OK, "device status");

    int32_t *g_idx = malloc(TK * 4), *g_slot = malloc(TK * 4), *g_counts = malloc((size_t)E * 4),
            *g_offsets = malloc((size_t)(E + 1) * 4), *g_rank = malloc((size_t)R * 4), g_drop = 0,
            *g_src = malloc(EC * 4);
    float *g_w = malloc(TK * 4), *g_scale = fp8 ? malloc(EC * nb * 4) : NULL;
    uint8_t *g_recv = malloc(ECH * 2);
    uint16_t *g_out = malloc(TH * 2);
    CUDA(cudaMemcpy(g_idx, d_idx, TK * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_slot, d_slot, TK * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_w, d_w, TK * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_counts, d_counts, (size_t)E * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_offsets, d_offsets, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_rank, d_rank, (size_t)R * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&g_drop, d_drop, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_src, d_src, EC * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_recv, d_recv, ECH * (fp8 ? 1 : 2), cudaMemcpyDeviceToHost));
    if (fp8) CUDA(cudaMemcpy(g_scale, d_scale, EC * nb * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(g_out, d_out, TH * 2, cudaMemcpyDeviceToHost));

    /* the oracle on the same host inputs */
    int32_t *o_idx = malloc(TK * 4), *o_slot = malloc(TK * 4), *o_counts = malloc((size_t)E * 4),
            *o_offsets = malloc((size_t)(E + 1) * 4), *o_rank = malloc((size_t)R * 4), o_drop = 0,
            *o_src = calloc(EC, 4);
    float *o_w = malloc(TK * 4), *o_scale = fp8 ? calloc(EC * nb, 4) : NULL;
    uint8_t *o_recv = calloc(ECH, 2);
    uint16_t *o_y = calloc(ECH, 2), *o_out = malloc(TH * 2);
    CHECK(oracle_route(T, E, k, logits, o_idx, o_w, NULL) == 0, "oracle_route");
    CHECK(oracle_count(T, E, k, R, C, o_idx, o_counts, o_offsets, o_slot, o_rank, &o_drop) == 0, "oracle_count");
    if (fp8)
        CHECK(oracle_dispatch_fp8(T, H, E, k, C, x, o_idx, o_slot, o_recv, o_scale, o_src) == 0, "oracle_dispatch");
    else
        CHECK(oracle_dispatch_bf16(T, H, E, k, C, x, o_idx, o_slot, (uint16_t *)o_recv, o_src) == 0, "oracle_dispatch");
    CHECK(oracle_expert_synthetic(H, E, C, fp8, o_recv, o_scale, o_counts, s, o_y) == 0, "oracle_expert");
    CHECK(oracle_combine(T, H, E, k, C, o_y, o_idx, o_w, o_slot, o_out) == 0, "oracle_combine");

    CHECK(memcmp(g_idx, o_idx, TK * 4) == 0, "topk_idx");
    CHECK(memcmp(g_slot, o_slot, TK * 4) == 0, "slot");
    CHECK(memcmp(g_counts, o_counts, (size_t)E * 4) == 0, "counts");
    CHECK(memcmp(g_offsets, o_offsets, (size_t)(E + 1) * 4) == 0, "offsets");
    CHECK(memcmp(g_rank, o_rank, (size_t)R * 4) == 0, "rank_counts");
    CHECK(g_drop == o_drop, "dropped");
    for (size_t i = 0; i < TK; ++i)
        CHECK(fabs((double)g_w[i] - o_w[i]) <= 1e-6 * fabs((double)o_w[i]), "topk_w[%zu]", i);
    const size_t rowb = (size_t)H * (fp8 ? 1 : 2);
    for (int32_t e = 0; e < E; ++e) {
        const int32_t kept = o_counts[e] < C ? o_counts[e] : C;
        for (int32_t r = 0; r < kept; ++r) {
            const size_t row = (size_t)e * C + r;
            CHECK(memcmp(g_recv + row * rowb, o_recv + row * rowb, rowb) == 0, "recv row (%d, %d)", e, r);
            CHECK(g_src[row] == o_src[row], "recv_src (%d, %d)", e, r);
            if (fp8) CHECK(memcmp(g_scale + row * nb, o_scale + row * nb, (size_t)nb * 4) == 0, "scale (%d, %d)", e, r);
        }
    }
    int32_t worst = 0;
    for (size_t i = 0; i < TH; ++i) {
        const int32_t d = abs(ordered(g_out[i]) - ordered(o_out[i]));
        if (d > worst) worst = d;
    }
    CHECK(worst <= 1, "combine differs by %d bf16 ulps", worst);

    /* the allocation-free route gives the same outputs */
    CUDA(cudaMemset(d_slot, 0x7F, TK * 4));
    MOE(moe_route_noalloc(&p, d_logits, d_idx, d_w, d_counts, d_offsets, d_slot, d_rank, d_drop, st));
    CUDA(cudaStreamSynchronize(st));
    int32_t *n_slot = malloc(TK * 4);
    CUDA(cudaMemcpy(n_slot, d_slot, TK * 4, cudaMemcpyDeviceToHost));
    CHECK(memcmp(n_slot, o_slot, TK * 4) == 0, "noalloc slot");

    printf("case T=%d H=%d E=%d k=%d %s: combine max %d ulp\n", T, H, E, k, fp8 ? "fp8" : "bf16", worst);
    CUDA(cudaStreamDestroy(st));
    void *dev[] = {d_x, d_recv, d_y, d_out, d_logits, d_w, d_s, d_scale, d_idx, d_slot, d_counts, d_offsets,
                   d_rank, d_drop, d_src, d_ws};
    for (size_t i = 0; i < sizeof dev / sizeof dev[0]; ++i)
        if (dev[i]) CUDA(cudaFree(dev[i]));
    void *host[] = {x, logits, s, g_idx, g_slot, g_counts, g_offsets, g_rank, g_src, g_w, g_scale, g_recv, g_out,
                    o_idx, o_slot, o_counts, o_offsets, o_rank, o_src, o_w, o_scale, o_recv, o_y, o_out, n_slot};
    for (size_t i = 0; i < sizeof host / sizeof host[0]; ++i) free(host[i]);
}

int main(void) {
    run_case(200, 512, 16, 4, 4, 64, 0, 11);      /* bf16, ragged tiles */
    run_case(300, 1024, 64, 6, 8, 32, 1, 12);     /* fp8, capacity overflow */
    if (failures) {
        fprintf(stderr, "%d checks failed\n", failures);
        return 1;
    }
    printf("c abi ok\n");
    return 0;
}
