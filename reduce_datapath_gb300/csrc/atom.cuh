// atom.cuh -- the Atom datapath for sm_103a: the two data-movement primitives of
// the page "Purlin: Separating Orchestration from the Datapath of Collectives"
// (abstract: Atom "implements two key data movement primitives for collectives:
// copy and reduce"; Figure 1: the Atom "deals only with how bytes move on a given
// GPU generation").
//
// On one GB300 every rank buffer is in local HBM, so both primitives are
// streaming HBM kernels: coalesced 16- or 32-byte accesses per thread (256-bit
// ld/st.global.v8 are native on this generation), L1 bypassed (each byte is
// touched once), and for sums a binary32 accumulator per element folded in rank
// order 0..R-1 and rounded once to the output type with round-to-nearest-even.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "plan.h"
#if defined(PURLIN_CHECKED)
#include "purlin.h"
#endif

namespace purlin {
namespace atom {

// ------------------------------------------------------------ checked builds
// With PURLIN_CHECKED every global access below is first tested against the
// launch's address ranges (CheckRanges, copied into shared memory when the
// kernel starts): one outside all of them is skipped (a load returns zeros),
// and the kernel records PURLIN_ERR_BOUNDS and the first such address (a
// misaligned access too, which the kernels never make).  A store must lie
// inside a range.  A load of a block aligned to its size need
// only hold a byte of one: the shifted bodies read the aligned blocks around a
// segment's ends, which stay within the pages the buffer lies in, while a
// block wholly outside every buffer is still caught.  A debug build for tests;
// the product build compiles none of it.
#if defined(PURLIN_CHECKED)
static __shared__ CheckRanges s_check;
static __shared__ int* s_check_status;

__device__ __forceinline__ void check_begin(const CheckRanges& c, int* status)
{
    if (threadIdx.x == 0) {
        s_check = c;
        s_check_status = status;
    }
    __syncthreads();
}

// bytes at p, which must be aligned to `align` (a misaligned access is
// reported rather than made); block: an aligned block that need only hold a
// byte of a range.
static __device__ __noinline__ bool access_ok(const void* p, uint32_t bytes, uint32_t align,
                                              bool block)
{
    const uint64_t a = reinterpret_cast<uint64_t>(p);
    const uint64_t e = a + bytes;
    const bool aligned = (a & (uint64_t)(align - 1)) == 0;
    for (uint32_t i = 0; aligned && i < s_check.n; ++i) {
        if (block ? (a < s_check.hi[i] && e > s_check.lo[i])
                  : (a >= s_check.lo[i] && e <= s_check.hi[i] && e >= a))
            return true;
    }
    atomicCAS(s_check_status, 0, (int)PURLIN_ERR_BOUNDS);
    if (s_check.bad) atomicCAS(s_check.bad, 0ull, (unsigned long long)a);
    return false;
}
#define PURLIN_CHECK_BEGIN(params) ::purlin::atom::check_begin((params).check, (params).status)
#define PURLIN_CHECK_LOAD(p, bytes, zero) \
    if (!::purlin::atom::access_ok((p), (bytes), (bytes), true)) { zero; return; }
#define PURLIN_CHECK_STORE(p, bytes) \
    if (!::purlin::atom::access_ok((p), (bytes), (bytes), false)) return;
#else
#define PURLIN_CHECK_BEGIN(params) ((void)0)
#define PURLIN_CHECK_LOAD(p, bytes, zero)
#define PURLIN_CHECK_STORE(p, bytes)
#endif

// ---------------------------------------------------------------- raw accesses

template <int BYTES> struct Vec;
template <> struct Vec<16> { uint32_t w[4]; };
template <> struct Vec<32> { uint32_t w[8]; };

// Loads skip L1 allocation: every source byte is read exactly once.
__device__ __forceinline__ void load(Vec<16>& v, const char* p)
{
    PURLIN_CHECK_LOAD(p, 16, v = Vec<16>{})
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
}

__device__ __forceinline__ void load(Vec<32>& v, const char* p)
{
    PURLIN_CHECK_LOAD(p, 32, v = Vec<32>{})
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

__device__ __forceinline__ void store(char* p, const Vec<16>& v)
{
    PURLIN_CHECK_STORE(p, 16)
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

__device__ __forceinline__ void store(char* p, const Vec<32>& v)
{
    PURLIN_CHECK_STORE(p, 32)
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]),
                    "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}

// L2 eviction priority for a whole launch, as a cache-policy operand
// (createpolicy): a stream read or written exactly once can be marked
// evict-first so that it does not push out lines another stream will reuse.
__device__ __forceinline__ uint64_t l2_policy(uint32_t kind)
{
    uint64_t pol;
    if (kind == kL2EvictFirst)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else if (kind == kL2EvictLast)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void load(Vec<16>& v, const char* p, uint64_t pol)
{
    PURLIN_CHECK_LOAD(p, 16, v = Vec<16>{})
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p), "l"(pol));
}

__device__ __forceinline__ void load(Vec<32>& v, const char* p, uint64_t pol)
{
    PURLIN_CHECK_LOAD(p, 32, v = Vec<32>{})
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7},"
                 " [%8], %9;"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p), "l"(pol));
}

__device__ __forceinline__ void store(char* p, const Vec<16>& v, uint64_t pol)
{
    PURLIN_CHECK_STORE(p, 16)
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void store(char* p, const Vec<32>& v, uint64_t pol)
{
    PURLIN_CHECK_STORE(p, 32)
    asm volatile("st.global.L2::cache_hint.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]),
                    "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7]), "l"(pol)
                 : "memory");
}

// Loads of data another CTA wrote during this kernel (the SNAC staging ring):
// cached in L2 only (.cg), so no stale L1 line can be returned.
__device__ __forceinline__ void load_cg(Vec<16>& v, const char* p)
{
    PURLIN_CHECK_LOAD(p, 16, v = Vec<16>{})
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
}

__device__ __forceinline__ void load_cg(Vec<32>& v, const char* p)
{
    PURLIN_CHECK_LOAD(p, 32, v = Vec<32>{})
    asm volatile("ld.global.cg.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

// --------------------------------------------------------- access units
// A copy moves bytes in units of 1..32 bytes (the widest alignment the source
// and destination share); vectors are 16 or 32 bytes.

template <int BYTES> struct Unit { Vec<BYTES> v; };
template <> struct Unit<1> { uint8_t v; };
template <> struct Unit<2> { uint16_t v; };
template <> struct Unit<4> { uint32_t v; };
template <> struct Unit<8> { uint2 v; };

// CG = true: L2-only load (staging ring); false: L1-bypassing load (sources).
template <int BYTES, bool CG = false>
__device__ __forceinline__ void load_unit(Unit<BYTES>& u, const char* p)
{
    PURLIN_CHECK_LOAD(p, BYTES, u = Unit<BYTES>{})
    if constexpr (BYTES >= 16) {
        if constexpr (CG) load_cg(u.v, p);
        else load(u.v, p);
    } else if constexpr (CG) {
        if constexpr (BYTES == 8)
            asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(u.v.x), "=r"(u.v.y) : "l"(p));
        else if constexpr (BYTES == 4)
            asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(u.v) : "l"(p));
        else if constexpr (BYTES == 2)
            asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(u.v) : "l"(p));
        else {
            uint16_t t;
            asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(t) : "l"(p));
            u.v = (uint8_t)t;
        }
    } else {
        if constexpr (BYTES == 8) u.v = *reinterpret_cast<const uint2*>(p);
        else if constexpr (BYTES == 4) u.v = *reinterpret_cast<const uint32_t*>(p);
        else if constexpr (BYTES == 2) u.v = *reinterpret_cast<const uint16_t*>(p);
        else u.v = *reinterpret_cast<const uint8_t*>(p);
    }
}

template <int BYTES>
__device__ __forceinline__ void store_unit(char* p, const Unit<BYTES>& u)
{
    PURLIN_CHECK_STORE(p, BYTES)
    if constexpr (BYTES >= 16) store(p, u.v);
    else if constexpr (BYTES == 8) *reinterpret_cast<uint2*>(p) = u.v;
    else if constexpr (BYTES == 4) *reinterpret_cast<uint32_t*>(p) = u.v;
    else if constexpr (BYTES == 2) *reinterpret_cast<uint16_t*>(p) = u.v;
    else *reinterpret_cast<uint8_t*>(p) = u.v;
}

// ------------------------------------------------------------ element codecs
// A 32-bit word holds one binary32 or two 16-bit values (low half first).

struct F32 {
    static constexpr int kPerWord = 1;
    static constexpr int kBytes = 4;
    __device__ static float widen(uint32_t w, int) { return __uint_as_float(w); }
    __device__ static uint32_t narrow(const float* f) { return __float_as_uint(f[0]); }
    __device__ static float load1(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 4, 4, false)) return 0.0f;
#endif
        return *reinterpret_cast<const float*>(p);
    }
    __device__ static float load1_cg(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 4, 4, false)) return 0.0f;
#endif
        float f;
        asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(f) : "l"(p));
        return f;
    }
    __device__ static void store1(char* p, float f)
    {
        PURLIN_CHECK_STORE(p, 4)
        *reinterpret_cast<float*>(p) = f;
    }
};

struct BF16 {
    static constexpr int kPerWord = 2;
    static constexpr int kBytes = 2;
    // bfloat16 -> binary32 is exact: the 16 bits become the high half.
    __device__ static float widen(uint32_t w, int half)
    {
        return __uint_as_float(half ? (w & 0xffff0000u) : (w << 16));
    }
    // binary32 pair -> bfloat16x2, round to nearest even (cvt.rn).
    __device__ static uint32_t narrow(const float* f)
    {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f[1]), "f"(f[0]));
        return r;
    }
    __device__ static float load1(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 2, 2, false)) return 0.0f;
#endif
        return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
    }
    __device__ static float load1_cg(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 2, 2, false)) return 0.0f;
#endif
        uint16_t h;
        asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p));
        return __uint_as_float((uint32_t)h << 16);
    }
    __device__ static void store1(char* p, float f)
    {
        PURLIN_CHECK_STORE(p, 2)
        float two[2] = {f, 0.0f};
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)(narrow(two) & 0xffffu);
    }
};

struct F16 {
    static constexpr int kPerWord = 2;
    static constexpr int kBytes = 2;
    __device__ static float widen(uint32_t w, int half)
    {
        return __half2float(__ushort_as_half((unsigned short)(half ? (w >> 16) : (w & 0xffffu))));
    }
    __device__ static uint32_t narrow(const float* f)
    {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f[1]), "f"(f[0]));
        return r;
    }
    __device__ static float load1(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 2, 2, false)) return 0.0f;
#endif
        return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(p)));
    }
    __device__ static float load1_cg(const char* p)
    {
#if defined(PURLIN_CHECKED)
        if (!access_ok(p, 2, 2, false)) return 0.0f;
#endif
        unsigned short h;
        asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p));
        return __half2float(__ushort_as_half(h));
    }
    __device__ static void store1(char* p, float f)
    {
        PURLIN_CHECK_STORE(p, 2)
        float two[2] = {f, 0.0f};
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)(narrow(two) & 0xffffu);
    }
};

// ------------------------------------------------------------------ the fold
// ORDER 0: left fold over ranks 0..R-1, starting from rank 0's value.
// ORDER 1: pairwise over ranks, ((x0+x1)+(x2+x3))+((x4+x5)+(x6+x7)); an odd
//          last value moves up a level unchanged.
// __fadd_rn keeps every add a separately rounded IEEE binary32 add.

template <int ORDER, int N>
__device__ __forceinline__ float fold(float (&v)[N], int R)
{
    static_assert(N <= kMaxRanks, "at most kMaxRanks values");
    if (ORDER == 0) {
        float acc = v[0];
#pragma unroll
        for (int r = 1; r < N; ++r)
            if (r < R) acc = __fadd_rn(acc, v[r]);
        return acc;
    } else {
        int live = R;
#pragma unroll
        for (int level = 0; level < 3; ++level) {
#pragma unroll
            for (int p = 0; p < N / 2; ++p) {
                if (2 * p + 1 < live) v[p] = __fadd_rn(v[2 * p], v[2 * p + 1]);
                else if (2 * p < live) v[p] = v[2 * p];
            }
            live = (live + 1) >> 1;
        }
        return v[0];
    }
}

// Atom::reduce of one vector unit: R source vectors (R <= NSRC) -> one output
// vector.
template <typename T, int ORDER, int BYTES, int NSRC>
__device__ __forceinline__ void reduce_unit(const Vec<BYTES> (&src)[NSRC], int R,
                                            Vec<BYTES>& dst)
{
    constexpr int W = BYTES / 4;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        float out[2];
#pragma unroll
        for (int h = 0; h < T::kPerWord; ++h) {
            float v[NSRC];
#pragma unroll
            for (int r = 0; r < NSRC; ++r) v[r] = (r < R) ? T::widen(src[r].w[w], h) : 0.0f;
            out[h] = fold<ORDER>(v, R);
        }
        dst.w[w] = T::narrow(out);
    }
}

}  // namespace atom
}  // namespace purlin
