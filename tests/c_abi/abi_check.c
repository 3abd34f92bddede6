/*
 * abi_check.c -- the C ABI used from plain C99, with no Python in between.
 *
 *   abi_check plan   host only: plan an AllGather with purlin_plan_segments and
 *                    check that the segments cover every output byte once.
 *   abi_check gpu    create a handle for 4 ranks, AllReduce fp32 integer values
 *                    (sums are exact in any order) and compare with the sums
 *                    computed here; then ReduceScatter + AllGather must equal it;
 *                    then the AllReduce kept as a plan and launched twice.
 * Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

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

int main(int argc, char** argv)
{
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
        int rc = gpu_check();
        printf("gpu check: %d\n", rc);
        return rc;
    }
    int rc = plan_check();
    printf("plan check: %d\n", rc);
    return rc;
}
