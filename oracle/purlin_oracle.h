/*
 * purlin_oracle.h -- prototypes of the CPU oracle for the Purlin collectives.
 *
 * TEST INFRASTRUCTURE ONLY.  This header belongs to the oracle and to nothing
 * else: the CUDA library does not include it, and the oracle does not include
 * any header of the CUDA library.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load the oracle.
 *
 * Page cited throughout: "Purlin: Separating Orchestration from the Datapath
 * of Collectives" (figure and table captions; abstract).
 *
 * Conventions (all functions):
 *   R          number of ranks, 1..64.
 *   x[r]/in[r] host pointer to rank r's input buffer.
 *   y[k]/out[j] host pointer to rank k's (j's) output buffer.
 *   counts, displacements are in ELEMENTS.  A NULL displacement array means
 *   "packed": partition k starts at the sum of the counts before it.
 *   dtype      ORACLE_F32, ORACLE_BF16 or ORACLE_F16 (raw 16-bit words).
 *   Return 0 on success, -1 on an argument the oracle does not accept.
 */
#ifndef PURLIN_ORACLE_H
#define PURLIN_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* Scalar codecs, written from the IEEE 754 binary16/binary32 and bfloat16
 * definitions (round to nearest, ties to even; no flush of subnormals). */
float    oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);
float    oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_f16(float f);

/* Array forms of the codecs, for the tests that pin them. */
void oracle_bf16_to_f32_n(const uint16_t* h, float* f, size_t n);
void oracle_f32_to_bf16_n(const float* f, uint16_t* h, size_t n);
void oracle_f16_to_f32_n(const uint16_t* h, float* f, size_t n);
void oracle_f32_to_f16_n(const float* f, uint16_t* h, size_t n);

/* ReduceScatter(V): y_k[i] = x_0[d_k+i] + x_1[d_k+i] + ... + x_{R-1}[d_k+i],
 * accumulated in binary32 in rank order 0..R-1, rounded once to dtype. */
int oracle_reduce_scatter(int R, const void* const* x, void* const* y,
                          const uint64_t* recv_counts, const uint64_t* in_displs,
                          int dtype);

/* AllGather(V): out_j[D_k + i] = in_k[i] for every j and k (rank order). */
int oracle_all_gather(int R, const void* const* in, void* const* out,
                      const uint64_t* counts, const uint64_t* out_displs,
                      size_t elem_bytes);

/* AllReduce: out_j[i] = x_0[i] + ... + x_{R-1}[i] for every j, same
 * accumulation and rounding as ReduceScatter. */
int oracle_all_reduce(int R, const void* const* x, void* const* out,
                      uint64_t count, int dtype);

/* AllToAll(V): out_j[rd[j][s] + i] = in_s[sd[s][j] + i], i < C[s][j].
 * send_counts and send_displs are R*R arrays indexed [s*R + j];
 * recv_displs is indexed [j*R + s]. */
int oracle_all_to_all_v(int R, const void* const* in, void* const* out,
                        const uint64_t* send_counts, const uint64_t* send_displs,
                        const uint64_t* recv_displs, size_t elem_bytes);

/* ReduceScatter(V) with the pairwise (tree) rank order instead of 0..R-1:
 * at each level, neighbours (2i, 2i+1) are added and an odd last value is
 * carried up unchanged. */
int oracle_reduce_scatter_tree(int R, const void* const* x, void* const* y,
                               const uint64_t* recv_counts, const uint64_t* in_displs,
                               int dtype);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_ORACLE_H */
