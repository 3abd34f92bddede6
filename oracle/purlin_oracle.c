/*
 * purlin_oracle.c -- a plain, slow CPU oracle for the layout semantics of the
 * Purlin collectives (ReduceScatter(V), AllGather(V), AllReduce, AllToAll(V)).
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never links, loads or calls this
 * file, and this file shares no code, header, table or helper with it.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may use it.
 *
 * Source of the semantics: the page "Purlin: Separating Orchestration from the
 * Datapath of Collectives":
 *   - Abstract: a collective is "a naming of an input and output layout and a
 *     copy or reduction operation".
 *   - Figure 4 (layouts on three ranks): ReduceScatter sums partition k of every
 *     input into y_k at rank k; AllGather puts every y_k, in rank order, at every
 *     rank; AllToAll gives rank j partition j of every source, in source order.
 *   - Figure 6 (composed AllReduce): AllReduce = AllGather after ReduceScatter.
 *   - Table 2: "(V)" marks the variable-length variant of a collective.
 * The pages do not fix the arithmetic of the reduction.  The reading taken here:
 * every output element is a left fold over ranks 0..R-1 in IEEE binary32
 * (round to nearest even), starting from rank 0's value, rounded ONCE to the
 * output type with round-to-nearest-even; subnormals are kept.
 *
 * Parity status: every function here is pinned by tests outside this file
 * (hand-worked examples, closed forms, invariants, library codecs); none is
 * "parity unpinned".
 *
 * Build: plain C99, no fast-math, no FMA contraction (there are no multiplies in
 * the reductions, but -ffp-contract=off keeps it so).
 */
#include "purlin_oracle.h"

#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar codecs                                                             */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* bfloat16 is the upper half of a binary32 word, so widening is a shift. */
float oracle_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even.  The bfloat16 values are
 * exactly the binary32 values whose low 16 bits are zero; the nearest one is the
 * truncation, or the truncation plus one unit of the kept part when the dropped
 * half-word is above one half (or exactly one half and the kept part is odd).
 * The carry runs into the exponent field, which also rounds the largest finite
 * values up to infinity as the standard requires.  A NaN stays a (quiet) NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* 2^e for small |e|, built exactly by repeated halving/doubling. */
static float pow2f(int e)
{
    float p = 1.0f;
    for (; e > 0; --e) p *= 2.0f;
    for (; e < 0; ++e) p *= 0.5f;
    return p;
}

/* binary16 -> binary32 (exact).  Fields: 1 sign, 5 exponent (bias 15), 10
 * fraction.  Exponent 0 holds zero and subnormals (fraction * 2^-24), exponent
 * 31 holds infinities and NaNs. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float mag;
    if (e == 0)
        mag = (float)m * pow2f(-24);
    else if (e == 31)
        mag = m ? f32_from_bits(0x7fc00000u) : f32_from_bits(0x7f800000u);
    else
        mag = (float)(m + 1024) * pow2f(e - 25);
    return sign ? -mag : mag;
}

/* Position of the highest set bit of a non-zero word. */
static int top_bit(uint32_t v)
{
    int b = -1;
    while (v) { v >>= 1; ++b; }
    return b;
}

/* binary32 -> binary16, round to nearest, ties to even.
 * Write |f| = M * 2^E with M an integer below 2^24.  Near |f| the binary16
 * values are spaced 2^q apart, q = floor(log2 |f|) - 10, but never closer than
 * the subnormal spacing 2^-24.  Rounding |f| / 2^q to the nearest integer n
 * (ties to even) gives the result n * 2^q, and its encoding is
 * ((q + 24) << 10) + n: for q = -24 the encoding is n itself (subnormals, and
 * n = 1024..2048 falls into the first normal binades), and for larger q,
 * n in [1024, 2048] puts the exponent field at q + 25 with fraction n - 1024
 * (n = 2048 carries into the next binade).  Encodings at or above 0x7c00 are
 * infinity. */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u = bits_from_f32(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);
    if (a == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);
    if (a == 0) return sign;

    uint32_t M;
    int E;
    int field = (int)(a >> 23);
    if (field == 0) { M = a & 0x7fffffu; E = -149; }
    else { M = (a & 0x7fffffu) | 0x800000u; E = field - 150; }

    int q = E + top_bit(M) - 10;
    if (q < -24) q = -24;
    int shift = q - E;

    uint32_t n;
    if (shift <= 0) {
        n = M << (-shift);
    } else if (shift > 25) {
        n = 0;                       /* M < 2^24, so |f| / 2^q < 1/2 */
    } else {
        uint32_t kept = M >> shift;
        uint32_t rest = M & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        n = kept + ((rest > half || (rest == half && (kept & 1u))) ? 1u : 0u);
    }
    uint32_t enc = ((uint32_t)(q + 24) << 10) + n;
    if (enc > 0x7c00u) enc = 0x7c00u;
    return (uint16_t)(sign | enc);
}

void oracle_bf16_to_f32_n(const uint16_t* h, float* f, size_t n)
{ for (size_t i = 0; i < n; ++i) f[i] = oracle_bf16_to_f32(h[i]); }
void oracle_f32_to_bf16_n(const float* f, uint16_t* h, size_t n)
{ for (size_t i = 0; i < n; ++i) h[i] = oracle_f32_to_bf16(f[i]); }
void oracle_f16_to_f32_n(const uint16_t* h, float* f, size_t n)
{ for (size_t i = 0; i < n; ++i) f[i] = oracle_f16_to_f32(h[i]); }
void oracle_f32_to_f16_n(const float* f, uint16_t* h, size_t n)
{ for (size_t i = 0; i < n; ++i) h[i] = oracle_f32_to_f16(f[i]); }

/* ------------------------------------------------------------------------ */
/* Element access                                                            */
/* ------------------------------------------------------------------------ */

static int dtype_ok(int dtype)
{ return dtype == ORACLE_F32 || dtype == ORACLE_BF16 || dtype == ORACLE_F16; }

static float load_elem(const void* base, uint64_t i, int dtype)
{
    if (dtype == ORACLE_F32) return ((const float*)base)[i];
    if (dtype == ORACLE_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
    return oracle_f16_to_f32(((const uint16_t*)base)[i]);
}

static void store_elem(void* base, uint64_t i, float v, int dtype)
{
    if (dtype == ORACLE_F32) ((float*)base)[i] = v;
    else if (dtype == ORACLE_BF16) ((uint16_t*)base)[i] = oracle_f32_to_bf16(v);
    else ((uint16_t*)base)[i] = oracle_f32_to_f16(v);
}

/* Partition k starts at displs[k], or, with no displacements given, right after
 * partitions 0..k-1 (Figure 4 lays partitions out in rank order). */
static uint64_t start_of(const uint64_t* counts, const uint64_t* displs, int k)
{
    if (displs) return displs[k];
    uint64_t s = 0;
    for (int m = 0; m < k; ++m) s += counts[m];
    return s;
}

/* Left fold over ranks 0..R-1 of element `at` in binary32. */
static float fold_ranks(int R, const void* const* x, uint64_t at, int dtype)
{
    float acc = load_elem(x[0], at, dtype);
    for (int r = 1; r < R; ++r)
        acc = acc + load_elem(x[r], at, dtype);
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Collectives                                                               */
/* ------------------------------------------------------------------------ */

/* Figure 4 (top): partition k of every input is summed into y_k at rank k. */
int oracle_reduce_scatter(int R, const void* const* x, void* const* y,
                          const uint64_t* recv_counts, const uint64_t* in_displs,
                          int dtype)
{
    if (R < 1 || R > 64 || !dtype_ok(dtype) || !recv_counts) return -1;
    for (int k = 0; k < R; ++k) {
        uint64_t d = start_of(recv_counts, in_displs, k);
        for (uint64_t i = 0; i < recv_counts[k]; ++i)
            store_elem(y[k], i, fold_ranks(R, x, d + i, dtype), dtype);
    }
    return 0;
}

/* Figure 4 (top): every rank receives every y_k, placed in rank order. */
int oracle_all_gather(int R, const void* const* in, void* const* out,
                      const uint64_t* counts, const uint64_t* out_displs,
                      size_t elem_bytes)
{
    if (R < 1 || R > 64 || !counts || elem_bytes == 0) return -1;
    for (int j = 0; j < R; ++j)
        for (int k = 0; k < R; ++k) {
            uint64_t D = start_of(counts, out_displs, k);
            memcpy((char*)out[j] + D * elem_bytes, in[k], counts[k] * elem_bytes);
        }
    return 0;
}

/* Figure 6: AllReduce leaves the full reduced vector at every rank.  Written
 * from that definition directly (not as AllGather of ReduceScatter), so that
 * the composition can be tested as an independent invariant. */
int oracle_all_reduce(int R, const void* const* x, void* const* out,
                      uint64_t count, int dtype)
{
    if (R < 1 || R > 64 || !dtype_ok(dtype)) return -1;
    for (uint64_t i = 0; i < count; ++i) {
        float acc = fold_ranks(R, x, i, dtype);
        for (int j = 0; j < R; ++j)
            store_elem(out[j], i, acc, dtype);
    }
    return 0;
}

/* Figure 4 (bottom): rank j receives partition j of every source s, in source
 * order.  Counts are per (source, destination) pair for the (V) variant. */
int oracle_all_to_all_v(int R, const void* const* in, void* const* out,
                        const uint64_t* send_counts, const uint64_t* send_displs,
                        const uint64_t* recv_displs, size_t elem_bytes)
{
    if (R < 1 || R > 64 || !send_counts || elem_bytes == 0) return -1;
    for (int j = 0; j < R; ++j) {
        uint64_t packed_recv = 0;
        for (int s = 0; s < R; ++s) {
            uint64_t c = send_counts[(size_t)s * R + j];
            uint64_t sd = start_of(send_counts + (size_t)s * R,
                                   send_displs ? send_displs + (size_t)s * R : 0, j);
            uint64_t rd = recv_displs ? recv_displs[(size_t)j * R + s] : packed_recv;
            memcpy((char*)out[j] + rd * elem_bytes,
                   (const char*)in[s] + sd * elem_bytes, c * elem_bytes);
            packed_recv += c;
        }
    }
    return 0;
}

/* Pairwise rank order: ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7)) for
 * R = 8; an odd value at the end of a level moves up unchanged. */
int oracle_reduce_scatter_tree(int R, const void* const* x, void* const* y,
                               const uint64_t* recv_counts, const uint64_t* in_displs,
                               int dtype)
{
    if (R < 1 || R > 64 || !dtype_ok(dtype) || !recv_counts) return -1;
    float v[64];
    for (int k = 0; k < R; ++k) {
        uint64_t d = start_of(recv_counts, in_displs, k);
        for (uint64_t i = 0; i < recv_counts[k]; ++i) {
            for (int r = 0; r < R; ++r) v[r] = load_elem(x[r], d + i, dtype);
            int live = R;
            while (live > 1) {
                int next = 0;
                for (int p = 0; p + 1 < live; p += 2) v[next++] = v[p] + v[p + 1];
                if (live & 1) v[next++] = v[live - 1];
                live = next;
            }
            store_elem(y[k], i, v[0], dtype);
        }
    }
    return 0;
}
