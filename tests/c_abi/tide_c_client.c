/*
 * A plain C11 user of the library's C ABI (include/tide.h): no Python, no
 * C++.  Test infrastructure.
 *
 *   tide_c_client host   plans built without a GPU (host-only flag): slot
 *                        size and shard pieces of a ragged group against
 *                        hand-computed values (Section 2.1 geometry), the
 *                        error convention, and the host schedule planners
 *                        (Figure 6b's Latin square, Figure 5a's rounds).
 *   tide_c_client gpu    (built with -DTIDE_C_CLIENT_GPU, linked to the CUDA
 *                        runtime and to the CPU oracle): the reduce-scatter
 *                        fold and the placements on a ragged group of 4
 *                        virtual ranks, compared bit for bit with the oracle.
 *
 * Prints "OK" and exits 0 when every check holds; otherwise prints the first
 * failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tide.h"

#define CHECK(cond, ...)                                                 \
    do {                                                                 \
        if (!(cond)) {                                                   \
            fprintf(stderr, "check failed (%s:%d): ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                                \
            fprintf(stderr, "\n");                                       \
            exit(1);                                                     \
        }                                                                \
    } while (0)

enum { P = 3, WMAX = 8 };
/* A ragged group: (dim0, row_numel) = (10, 4), (2, 3), (7, 1). */
static const int64_t kDim0[P] = {10, 2, 7};
static const int64_t kRowNumel[P] = {4, 3, 1};

static void describe(int32_t world, const void *const ptrs[P][WMAX], tide_param_desc_t *desc)
{
    for (int p = 0; p < P; ++p) {
        desc[p].rank_base = ptrs[p];
        desc[p].dim0 = kDim0[p];
        desc[p].row_numel = kRowNumel[p];
        desc[p].shard_offset = -1;
    }
    (void)world;
}

static int host_checks(void)
{
    /* W = 3: R = (4, 1, 3); shards 16, 3, 3 elements at offsets 0, 16, 19; S = 22.
     * Rank 2 holds rows 8..9 of parameter 0 (8 real elements, 8 padding) and
     * no row of parameter 1 (3 padding). */
    const int32_t W = 3;
    const void *ptrs[P][WMAX];
    uintptr_t cur = 0x7f0000000000u;
    for (int p = 0; p < P; ++p)
        for (int u = 0; u < W; ++u, cur += 4096)
            ptrs[p][u] = (const void *)cur;
    tide_param_desc_t desc[P];
    describe(W, (const void *const(*)[WMAX])ptrs, desc);
    tide_plan_flags_t flags;
    memset(&flags, 0, sizeof flags);
    flags.debug = TIDE_DEBUG_HOST_ONLY;
    tide_plan_t *plan = NULL;
    tide_status_t st = tide_plan_build(W, P, desc, &flags, NULL, &plan);
    CHECK(st == TIDE_OK, "host-only plan: %s (%s)", tide_status_string(st), tide_last_error());
    CHECK(tide_plan_slot_numel(plan) == 22, "S = %lld, want 22", (long long)tide_plan_slot_numel(plan));
    CHECK(tide_plan_num_segments(plan) == P * W, "pieces");
    static const int64_t want_valid[P][3] = {{16, 16, 8}, {3, 3, 0}, {3, 3, 1}};
    static const int64_t want_dst[P] = {0, 16, 19};
    for (int p = 0; p < P; ++p)
        for (int r = 0; r < W; ++r) {
            tide_segment_t seg;
            CHECK(tide_plan_segment(plan, (int64_t)p * W + r, &seg) == TIDE_OK, "segment");
            const int64_t shard = p == 0 ? 16 : 3;
            CHECK(seg.param == p && seg.rank == r, "piece order");
            CHECK(seg.n_valid == want_valid[p][r] && seg.n_pad == shard - want_valid[p][r],
                  "piece (%d, %d): %lld valid + %lld padding", p, r, (long long)seg.n_valid, (long long)seg.n_pad);
            CHECK(seg.dst_elem == want_dst[p] && seg.src_elem == (int64_t)r * shard, "piece (%d, %d) offsets", p, r);
        }
    CHECK(tide_plan_destroy(plan) == TIDE_OK, "destroy");

    /* errors are status codes with a detail message */
    st = tide_plan_build(0, P, desc, &flags, NULL, &plan);
    CHECK(st == TIDE_ERR_INVALID_ARG && strlen(tide_last_error()) > 0, "world 0 must be INVALID_ARG");
    ptrs[1][2] = (const void *)((uintptr_t)ptrs[1][2] + 1);
    st = tide_plan_build(W, P, desc, &flags, NULL, &plan);
    CHECK(st == TIDE_ERR_ALIGNMENT, "odd gradient pointer must be ALIGNMENT, got %s", tide_status_string(st));
    CHECK(strcmp(tide_status_string(TIDE_ERR_TIMEOUT), "TIDE_ERR_TIMEOUT") == 0, "status string");

    /* Figure 6b (L = 4, M = 4): GPU 1 lands contributors C, D, A, B in sub-slices 0..3,
     * i.e. c = 3, 4 (own node), 1, 2. */
    static const int32_t want_c[4] = {3, 4, 1, 2};
    for (int32_t s = 0; s < 4; ++s) {
        const int32_t c = want_c[s], n = (0 - c % 4 + 4) % 4; /* destination node 0, contributor n */
        CHECK(tide_latin_square_gpu(s, 0, n, 4, 4) == 1, "Latin square, sub-slice %d", s);
    }
    /* Figure 5a: M = 5 takes three rounds forwarding 1, 2 and 1 shards. */
    int32_t count[8], step[8];
    CHECK(tide_bruck_schedule(5, count, step, 8) == 3, "rounds");
    CHECK(count[0] == 1 && count[1] == 2 && count[2] == 1 && step[2] == 4, "recursive doubling counts");
    /* Section 2.2, Equation (4): 36 slots, 128 CTAs in clusters of 4 -> (36 - 32) * 4 */
    CHECK(tide_corun_cta_budget(36, 128, 4) == 16, "co-run budget");
    CHECK(tide_corun_cta_budget(32, 128, 4) == 0 && tide_corun_cta_budget(0, 128, 4) == -1, "co-run budget edges");
    return 0;
}

#ifdef TIDE_C_CLIENT_GPU
#include <cuda_runtime.h>

/* The CPU oracle (tests only). */
int oracle_rs(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
              const uint16_t *const *grads, float alpha, int32_t accumulate, float *out, int64_t stride);
int oracle_ag(int32_t world, int32_t nparams, const int64_t *dim0, const int64_t *row_numel,
              const uint16_t *slots, int64_t stride, uint16_t *const *full);

#define CUDA_OK(call) CHECK((call) == cudaSuccess, "%s", #call)

static uint32_t lcg(uint32_t *s)
{
    *s = *s * 1664525u + 1013904223u;
    return *s;
}

/* A finite bf16 bit pattern of moderate magnitude (exponent 120..134). */
static uint16_t some_bf16(uint32_t *s)
{
    const uint32_t x = lcg(s);
    return (uint16_t)(((x >> 31) << 15) | ((120u + (x >> 8) % 15u) << 7) | (x & 0x7fu));
}

static int gpu_checks(void)
{
    const int32_t W = 4;
    const int64_t stride = 40; /* rank slot stride; S = 12 + 3 + 2 = 17 at W = 4 (checked below) */
    uint32_t seed = 12345u;
    uint16_t *h_grads[P][WMAX];
    void *d_grads[P][WMAX];
    const void *ptrs[P][WMAX];
    for (int p = 0; p < P; ++p)
        for (int u = 0; u < W; ++u) {
            const size_t n = (size_t)(kDim0[p] * kRowNumel[p]);
            h_grads[p][u] = (uint16_t *)malloc(n * 2);
            for (size_t j = 0; j < n; ++j)
                h_grads[p][u][j] = some_bf16(&seed);
            CUDA_OK(cudaMalloc(&d_grads[p][u], n * 2));
            CUDA_OK(cudaMemcpy(d_grads[p][u], h_grads[p][u], n * 2, cudaMemcpyHostToDevice));
            ptrs[p][u] = d_grads[p][u];
        }
    tide_param_desc_t desc[P];
    describe(W, (const void *const(*)[WMAX])ptrs, desc);
    tide_plan_t *plan = NULL;
    tide_status_t st = tide_plan_build(W, P, desc, NULL, NULL, &plan);
    CHECK(st == TIDE_OK, "plan: %s (%s)", tide_status_string(st), tide_last_error());
    const int64_t S = tide_plan_slot_numel(plan);
    CHECK(S <= stride, "S = %lld", (long long)S);

    /* reduce-scatter, alpha = 1/W, then accumulate a second one on top */
    float h_out[WMAX * 40], want[WMAX * 40];
    for (int i = 0; i < W * stride; ++i)
        h_out[i] = want[i] = 0.0f;
    float *d_out;
    CUDA_OK(cudaMalloc((void **)&d_out, sizeof h_out));
    CUDA_OK(cudaMemcpy(d_out, h_out, sizeof(float) * (size_t)(W * stride), cudaMemcpyHostToDevice));
    CHECK(tide_rs_fold(plan, d_out, stride, 0.25f, 0, NULL) == TIDE_OK, "fold");
    CHECK(tide_rs_fold(plan, d_out, stride, 1.0f, 1, NULL) == TIDE_OK, "fold, accumulate");
    CUDA_OK(cudaMemcpy(h_out, d_out, sizeof(float) * (size_t)(W * stride), cudaMemcpyDeviceToHost));
    CHECK(tide_last_device_status(plan, NULL) == TIDE_OK, "device status");
    /* the allocation-free fold on the same group: the same bits, and its own status word */
    float h_out2[WMAX * 40];
    float *d_out2;
    CUDA_OK(cudaMalloc((void **)&d_out2, sizeof h_out2));
    CUDA_OK(cudaMemset(d_out2, 0, sizeof(float) * (size_t)(W * stride)));
    CHECK(tide_rs_fold_noalloc(W, P, desc, d_out2, stride, 0.25f, 0, NULL) == TIDE_OK, "allocation-free fold");
    CHECK(tide_rs_fold_noalloc(W, P, desc, d_out2, stride, 1.0f, 1, NULL) == TIDE_OK, "allocation-free, accumulate");
    CUDA_OK(cudaMemcpy(h_out2, d_out2, sizeof(float) * (size_t)(W * stride), cudaMemcpyDeviceToHost));
    CHECK(tide_last_device_status(NULL, NULL) == TIDE_OK, "allocation-free fold's device status");
    const uint16_t *gp[P * WMAX];
    for (int p = 0; p < P; ++p)
        for (int u = 0; u < W; ++u)
            gp[p * W + u] = h_grads[p][u];
    CHECK(oracle_rs(W, P, kDim0, kRowNumel, gp, 0.25f, 0, want, stride) == 0, "oracle");
    CHECK(oracle_rs(W, P, kDim0, kRowNumel, gp, 1.0f, 1, want, stride) == 0, "oracle, accumulate");
    for (int r = 0; r < W; ++r) {
        CHECK(memcmp(h_out + r * stride, want + r * stride, sizeof(float) * (size_t)S) == 0,
              "fold differs from the oracle in rank slot %d", r);
        CHECK(memcmp(h_out2 + r * stride, want + r * stride, sizeof(float) * (size_t)S) == 0,
              "allocation-free fold differs from the oracle in rank slot %d", r);
    }

    /* placement on the SM kernel and on the copy engines */
    uint16_t h_slots[WMAX * 40];
    for (int i = 0; i < W * stride; ++i)
        h_slots[i] = some_bf16(&seed);
    void *d_slots;
    CUDA_OK(cudaMalloc(&d_slots, sizeof h_slots));
    CUDA_OK(cudaMemcpy(d_slots, h_slots, sizeof(uint16_t) * (size_t)(W * stride), cudaMemcpyHostToDevice));
    uint16_t *h_want[P], *h_full[P];
    void *d_full[P];
    for (int p = 0; p < P; ++p) {
        const size_t n = (size_t)(kDim0[p] * kRowNumel[p]);
        h_want[p] = (uint16_t *)malloc(n * 2);
        h_full[p] = (uint16_t *)malloc(n * 2);
        CUDA_OK(cudaMalloc(&d_full[p], n * 2));
    }
    CHECK(oracle_ag(W, P, kDim0, kRowNumel, h_slots, stride, h_want) == 0, "oracle placement");
    const int32_t modes[3] = {TIDE_AG_SM, TIDE_AG_CE_2D, TIDE_AG_CE_1D};
    for (int m = 0; m < 3; ++m) {
        for (int p = 0; p < P; ++p)
            CUDA_OK(cudaMemset(d_full[p], 0xff, (size_t)(kDim0[p] * kRowNumel[p]) * 2));
        CHECK(tide_ag_place(plan, d_slots, stride, d_full, modes[m], NULL) == TIDE_OK, "placement mode %d", m);
        CUDA_OK(cudaDeviceSynchronize());
        for (int p = 0; p < P; ++p) {
            const size_t n = (size_t)(kDim0[p] * kRowNumel[p]);
            CUDA_OK(cudaMemcpy(h_full[p], d_full[p], n * 2, cudaMemcpyDeviceToHost));
            CHECK(memcmp(h_full[p], h_want[p], n * 2) == 0, "placement mode %d differs, parameter %d", m, p);
        }
    }
    CHECK(tide_plan_destroy(plan) == TIDE_OK, "destroy");
    for (int p = 0; p < P; ++p) {
        for (int u = 0; u < W; ++u) {
            CUDA_OK(cudaFree(d_grads[p][u]));
            free(h_grads[p][u]);
        }
        CUDA_OK(cudaFree(d_full[p]));
        free(h_want[p]);
        free(h_full[p]);
    }
    CUDA_OK(cudaFree(d_out));
    CUDA_OK(cudaFree(d_out2));
    CUDA_OK(cudaFree(d_slots));
    return 0;
}
#endif

int main(int argc, char **argv)
{
    if (argc < 2) {
        fprintf(stderr, "usage: %s host|gpu\n", argv[0]);
        return 2;
    }
    if (strcmp(argv[1], "host") == 0) {
        host_checks();
    } else if (strcmp(argv[1], "gpu") == 0) {
#ifdef TIDE_C_CLIENT_GPU
        gpu_checks();
#else
        fprintf(stderr, "built without TIDE_C_CLIENT_GPU\n");
        return 2;
#endif
    } else {
        return 2;
    }
    printf("OK\n");
    return 0;
}
