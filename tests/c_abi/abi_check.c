/*
 * abi_check.c -- the C ABI used from plain C99, with no Python in between.
 *
 *   abi_check plan   host only: plan an AllGather with purlin_plan_segments and
 *                    check that the segments cover every output byte once.
 *   abi_check gpu    create a handle for 4 ranks, AllReduce fp32 integer values
 *                    (sums are exact in any order) and compare with the sums
 *                    computed here; then ReduceScatter + AllGather must equal it;
 *                    then the AllReduce kept as a plan and launched twice.
 *   abi_check cost   host time per call of an 8-rank bf16 AllReduce of 4 KiB per
 *                    rank, printed as one JSON line: planning alone
 *                    (purlin_plan_segments), recording a plan (begin, call, end,
 *                    destroy: layout and kernel parameters, nothing enqueued),
 *                    a direct call (planning + launch) and a recorded plan's
 *                    launch.
 * Exit status 0 on success.
 */
#define _POSIX_C_SOURCE 199309L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime_api.h>

#include "purlin.h"
#include "purlin_layout.h"

static int plan_check(void)
{
    enum { R = 3 };
    uint64_t in_addr[R] = {0x100000, 0x200000, 0x300000};
    uint64_t out_addr[R] = {0x400000, 0x500000, 0x600000};
    size_t counts[R] = {5, 0, 7};
    purlin_segment_t segs[32];
    int n = 0;
    uint32_t tiles = 0;
    if (purlin_plan_segments(PURLIN_COLL_ALL_GATHER, R, in_addr, out_addr, counts, NULL, NULL, 0,
                             PURLIN_F32, 32, segs, 32, &n, &tiles) != PURLIN_OK)
        return 1;
    /* packed AllGather: 12 elements = 48 bytes written to each of the 3 outputs */
    unsigned char seen[48];
    memset(seen, 0, sizeof seen);
    for (int i = 0; i < n; ++i) {
        if (segs[i].dst_rank != -1) return 2;
        for (uint64_t b = 0; b < segs[i].bytes; ++b) seen[segs[i].dst_off + b]++;
    }
    for (int b = 0; b < 48; ++b)
        if (seen[b] != 1) return 3;
    return purlin_version() >> 16 == 1 ? 0 : 4;
}

static int gpu_check(void)
{
    enum { R = 4, N = 10007 };
    float* host_in[R];
    void* din[R];
    void* dout[R];
    float* exact = (float*)malloc(N * sizeof(float));
    float* got = (float*)malloc(N * sizeof(float));
    if (!exact || !got) return 10;
    for (int i = 0; i < N; ++i) exact[i] = 0.0f;
    for (int r = 0; r < R; ++r) {
        host_in[r] = (float*)malloc(N * sizeof(float));
        if (!host_in[r]) return 10;
        for (int i = 0; i < N; ++i) {
            host_in[r][i] = (float)((i * 7 + r * 13) % 17 - 8);   /* integers in [-8, 8] */
            exact[i] += host_in[r][i];
        }
        if (cudaMalloc(&din[r], N * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&dout[r], N * sizeof(float)) != cudaSuccess)
            return 11;
        cudaMemcpy(din[r], host_in[r], N * sizeof(float), cudaMemcpyHostToDevice);
    }
    purlin_handle_t h = NULL;
    if (purlin_create(&h, R, 0, 0) != PURLIN_OK) return 12;
    if (purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_F32, PURLIN_OP_SUM, NULL) !=
        PURLIN_OK)
        return 13;
    if (cudaDeviceSynchronize() != cudaSuccess || purlin_query_status(h) != PURLIN_OK) return 14;
    for (int r = 0; r < R; ++r) {
        cudaMemcpy(got, dout[r], N * sizeof(float), cudaMemcpyDeviceToHost);
        if (memcmp(got, exact, N * sizeof(float)) != 0) return 15;
    }
    /* ReduceScatter into R pieces, then AllGather back: same vector */
    size_t counts[R];
    size_t left = N;
    for (int k = 0; k < R; ++k) { counts[k] = k < R - 1 ? N / R : left; left -= counts[k]; }
    void* piece[R];
    size_t off = 0;
    for (int k = 0; k < R; ++k) {
        if (cudaMalloc(&piece[k], counts[k] * sizeof(float) + 16) != cudaSuccess) return 16;
        off += counts[k];
    }
    if (purlin_reduce_scatter(h, (const void* const*)din, piece, counts, NULL, PURLIN_F32,
                              PURLIN_OP_SUM, NULL) != PURLIN_OK ||
        purlin_all_gather(h, (const void* const*)piece, dout, counts, NULL, PURLIN_F32, NULL) !=
            PURLIN_OK)
        return 17;
    if (cudaDeviceSynchronize() != cudaSuccess) return 18;
    for (int r = 0; r < R; ++r) {
        cudaMemcpy(got, dout[r], N * sizeof(float), cudaMemcpyDeviceToHost);
        if (memcmp(got, exact, N * sizeof(float)) != 0) return 19;
    }
    /* the AllReduce kept as a plan: recording enqueues nothing, each launch
       gives the exact sums again */
    purlin_plan_t plan = NULL;
    for (int r = 0; r < R; ++r) cudaMemset(dout[r], 0, N * sizeof(float));
    if (purlin_plan_begin(h) != PURLIN_OK ||
        purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_F32, PURLIN_OP_SUM, NULL) !=
            PURLIN_OK ||
        purlin_plan_end(h, &plan) != PURLIN_OK || plan == NULL)
        return 21;
    if (cudaDeviceSynchronize() != cudaSuccess) return 22;
    cudaMemcpy(got, dout[0], N * sizeof(float), cudaMemcpyDeviceToHost);
    for (int i = 0; i < N; ++i)
        if (got[i] != 0.0f) return 23;
    for (int rep = 0; rep < 2; ++rep) {
        if (purlin_plan_launch(plan, NULL) != PURLIN_OK) return 24;
        if (cudaDeviceSynchronize() != cudaSuccess || purlin_query_status(h) != PURLIN_OK)
            return 25;
        for (int r = 0; r < R; ++r) {
            cudaMemcpy(got, dout[r], N * sizeof(float), cudaMemcpyDeviceToHost);
            if (memcmp(got, exact, N * sizeof(float)) != 0) return 26;
        }
    }
    if (purlin_plan_destroy(plan) != PURLIN_OK) return 27;
    if (purlin_destroy(h) != PURLIN_OK) return 20;
    for (int r = 0; r < R; ++r) {
        cudaFree(din[r]);
        cudaFree(dout[r]);
        cudaFree(piece[r]);
        free(host_in[r]);
    }
    free(exact);
    free(got);
    return 0;
}

static double now_us(void)
{
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return t.tv_sec * 1e6 + t.tv_nsec * 1e-3;
}

static int cost_check(void)
{
    enum { R = 8, N = 2048, ITERS = 20000 };   /* 2048 bf16 = 4 KiB per rank */
    void* din[R];
    void* dout[R];
    uint64_t in_addr[R], out_addr[R];
    for (int r = 0; r < R; ++r) {
        if (cudaMalloc(&din[r], N * 2) != cudaSuccess || cudaMalloc(&dout[r], N * 2) != cudaSuccess)
            return 30;
        cudaMemset(din[r], 0, N * 2);
        in_addr[r] = (uint64_t)(uintptr_t)din[r];
        out_addr[r] = (uint64_t)(uintptr_t)dout[r];
    }
    purlin_segment_t segs[64];
    int nseg = 0;
    uint32_t tiles = 0;
    double t0 = now_us();
    for (int i = 0; i < ITERS; ++i)
        if (purlin_plan_segments(PURLIN_COLL_ALL_REDUCE, R, in_addr, out_addr, NULL, NULL, NULL, N,
                                 PURLIN_BF16, 32, segs, 64, &nseg, &tiles) != PURLIN_OK)
            return 31;
    const double plan_us = (now_us() - t0) / ITERS;

    purlin_handle_t h = NULL;
    if (purlin_create(&h, R, 0, 0) != PURLIN_OK) return 32;
    purlin_plan_t plan = NULL;
    for (int i = 0; i < 100; ++i)   /* warm-up: context, module, residency queries */
        if (purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_BF16, PURLIN_OP_SUM,
                              NULL) != PURLIN_OK)
            return 33;
    if (cudaDeviceSynchronize() != cudaSuccess) return 34;
    t0 = now_us();
    for (int i = 0; i < ITERS; ++i) {
        if (purlin_plan_begin(h) != PURLIN_OK ||
            purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_BF16, PURLIN_OP_SUM,
                              NULL) != PURLIN_OK ||
            purlin_plan_end(h, &plan) != PURLIN_OK || purlin_plan_destroy(plan) != PURLIN_OK)
            return 35;
    }
    const double record_us = (now_us() - t0) / ITERS;
    t0 = now_us();
    for (int i = 0; i < ITERS; ++i)
        if (purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_BF16, PURLIN_OP_SUM,
                              NULL) != PURLIN_OK)
            return 36;
    const double call_us = (now_us() - t0) / ITERS;
    if (cudaDeviceSynchronize() != cudaSuccess) return 37;
    if (purlin_plan_begin(h) != PURLIN_OK ||
        purlin_all_reduce(h, (const void* const*)din, dout, N, PURLIN_BF16, PURLIN_OP_SUM, NULL) !=
            PURLIN_OK ||
        purlin_plan_end(h, &plan) != PURLIN_OK)
        return 38;
    t0 = now_us();
    for (int i = 0; i < ITERS; ++i)
        if (purlin_plan_launch(plan, NULL) != PURLIN_OK) return 39;
    const double launch_us = (now_us() - t0) / ITERS;
    if (cudaDeviceSynchronize() != cudaSuccess || purlin_query_status(h) != PURLIN_OK) return 40;
    purlin_plan_destroy(plan);
    purlin_destroy(h);
    for (int r = 0; r < R; ++r) {
        cudaFree(din[r]);
        cudaFree(dout[r]);
    }
    printf("{\"R\": %d, \"bytes_per_rank\": %d, \"segments\": %d, \"plan_segments_us\": %.3f, "
           "\"record_plan_us\": %.3f, \"call_us\": %.3f, \"plan_launch_us\": %.3f, \"iters\": %d}\n",
           R, N * 2, nseg, plan_us, record_us, call_us, launch_us, ITERS);
    return 0;
}

int main(int argc, char** argv)
{
    if (argc > 1 && strcmp(argv[1], "cost") == 0) return cost_check();
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
        int rc = gpu_check();
        printf("gpu check: %d\n", rc);
        return rc;
    }
    int rc = plan_check();
    printf("plan check: %d\n", rc);
    return rc;
}
