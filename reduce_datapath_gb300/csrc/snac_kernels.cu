// snac_kernels.cu -- the SNAC (Stage, Notify, And Consume) protocol on one GPU.
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives":
//   - Abstract: SNAC is a shared orchestration protocol that derives
//     coordination from the collective's layouts, sitting above the Atom.
//   - Figure 6: in the composed AllReduce "all ranks stage chunks
//     incrementally"; rank k reduces chunks of partition k from all ranks while
//     gathering reduced chunks of other partitions.
//   - Figure 9 / Figure 16: staging serves "ordinary application buffers";
//     Figure 10: "Purlin-ZS omits staging" (zs_kernels.cu).
//   - Table 3: chunks sized to the bandwidth-delay product; Figure 11: pipeline
//     depth one to eight stages.
//
// One cooperative launch holds every role, so each waiting CTA's partner is
// resident.  Roles by blockIdx.x / channels:
//   0 producer(ch): for each of its steps, wait until its ring slot is free,
//     STAGE the step into the slot, NOTIFY (release).  It stages the step's
//     chunk of the source (copies), the R input chunks (sums, inputs staged),
//     or the chunk of y it reduces from the R inputs itself (sums, reduced
//     chunk staged).
//   1 consumer(ch): wait for the step's tag (acquire), CONSUME the slot: sum
//     the R staged chunks into the destination -- or, for AllReduce, into the
//     slot's y part -- or copy the staged chunk to its destination(s); then
//     free the slot.
//   2 gatherer(ch), AllReduce with inputs staged only: wait for the y tag, copy
//     the reduced chunk to all R outputs, free the y part.
// Steps are the layout's segments cut into chunks of `chunk` bytes per rank.
// Producers take steps from a device counter, and the producer records in the
// slot which step it staged.  A channel's n-th step sits in slot
// n % depth; a flag holds the tag (epoch << 32) | (n + 1).  The epoch lives in
// device memory (the last flag word): every CTA reads it when the kernel
// starts, and the last CTA to finish advances it (a completion counter in the
// word before it) and resets the step counter (the word before that), so each
// call -- also each replay of a captured CUDA graph -- runs with a fresh epoch
// and the flags never need resetting.  Every wait is bounded (time and
// iteration count) and watches the status word: on a timeout the waiter
// records PURLIN_ERR_TIMEOUT and every CTA leaves at its next wait.
#include "atom.cuh"
#include "internal.h"
#include "snac.h"
#include "zs_kernels.cuh"  // register realignment of shifted bodies

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace purlin {

namespace {

// kRS / kAR stage the R input chunks of a step and the consumer reduces them;
// kRSY / kARY reduce in the producer and stage the reduced chunk y, which the
// consumer copies to its destination (kRSY) or to all R outputs (kARY).
enum Kind : int { kRS = 0, kAG = 1, kAR = 2, kA2A = 3, kRSY = 4, kARY = 5 };
// Words per (channel, slot): the ready / free tags of the slot, the y-ready /
// y-free tags of its y part (three-role AllReduce), the step staged in the slot
// and the step whose reduced chunk sits in the y part.  Tags are
// (epoch << 32) | (n + 1) with epoch >= 1, so always >= 2^32; step words are
// always < 2^32; so a word one kind leaves behind can never release a wait of
// another kind on the same handle.
enum : int { kReady = 0, kFree = 1, kYReady = 2, kYFree = 3, kStepOf = 4, kYStepOf = 5,
             kFlagsPerSlot = 6 };
constexpr uint64_t kNoStep = 0xffffffffull;  // no step left; steps are < 2^32 - 1 (plan_into)

// Default chunk per rank per step, measured best on GB300 at 64 MiB per rank,
// depth 2, 64-thread role CTAs (event-timed, 20 launches; the time is not
// monotonic in the chunk, so each default is the best of a sweep):
//   - sums with the inputs staged put R (+ 1 for the AllReduce's y part) parts
//     in a slot and do best with a slot of about 48 KiB (ReduceScatter) or
//     72 KiB (AllReduce) whatever R: at R = 8 the ReduceScatter runs 176.0 us at
//     6 KiB (185.7 at 8, 231.0 at 12 KiB) and the AllReduce 264.4 us at 8 KiB
//     (285.1 at 12, 331.0 at 16); at R = 2 82.5 us at 16 KiB (100.6 at 6) and
//     118.1 us at 24 KiB (148.6 at 8); at R = 3 131.0 us at 12 KiB and 141.9 us
//     at 16 KiB; at R = 4 114.4 us at 12 KiB and 167.0 us at 16 KiB;
//   - sums with the reduced chunk staged put one part in a slot: ReduceScatter
//     117.9 us at 16 KiB (121.4 at 24, 127.0 at 32 KiB; 16 KiB is also best at
//     R = 2, 3 and 4), AllReduce 186.2 us at 12 KiB (188.2 at 16, 189.9 at 24);
//   - copies put one part in a slot: AllGather 104.7 us at 16 KiB (106.4 at 12,
//     108.7 at 24, 114.5 at 32 KiB), AllToAllV 241.3 us at 48 KiB (247.0 at 32,
//     254.1 at 64 KiB).
size_t default_chunk(Coll coll, int R, bool stage_y)
{
    const bool sum = coll == Coll::ReduceScatter || coll == Coll::AllReduce;
    if (stage_y && sum) return coll == Coll::ReduceScatter ? 16 * 1024 : 12 * 1024;
    const size_t k512 = 512;
    switch (coll) {
    case Coll::AllGather: return 16 * 1024;
    case Coll::AllToAllV: return 48 * 1024;
    case Coll::ReduceScatter:
        return std::min<size_t>(16 * 1024, (48 * 1024 / (size_t)R) / k512 * k512);
    default: return (72 * 1024 / (size_t)(R + 1)) / k512 * k512;
    }
}

// Widest unit of a launch: a sum launch holding a shifted body is planned
// with 16-byte units throughout (plan_into), so its kernel carries no 32-byte
// path (the shifted sums need the registers).
__host__ __device__ constexpr int snac_max_unit(int kind, bool shifted)
{
    return (shifted && kind != kAG && kind != kA2A) ? 4 : 5;
}

// Role CTAs of two warps, eight per SM (128 registers a thread, as 256-thread
// CTAs at two per SM have): more, narrower channels.  At 64 MiB per rank, R = 8,
// bf16, each kind at its best chunk, 256 / 128 / 64 / 32 threads per CTA:
// AllGather 115-120 / 109.8 / 104.7 / 104.1 us, AllReduce with the inputs staged
// 290 / 266.3 / 264.4 / 285.8, ReduceScatter with the inputs staged 185 / 174.7 /
// 176.0 / 185.7, AllToAllV 251 / 240.8 / 241.3 / 247.8.
constexpr int kSnacThreads = 64;
constexpr int kSnacCtasPerSm = 8;
constexpr int kDefaultDepth = 2;
constexpr int kMaxChannels = 640;
constexpr size_t kMinAutoChunk = 1024;

struct SnacParams {
    const char* in[kMaxRanks];
    char* out[kMaxRanks];
    char* staging;
    uint64_t* flags;
    int* status;
    uint64_t* epoch_word;    // device epoch of the last completed call
    uint32_t* done_word;     // CTAs of the running call that have finished
    unsigned long long* step_word;  // next step to hand out
    uint64_t timeout_ns;
    uint64_t max_spins;
    uint64_t chunk;        // bytes per rank per step (multiple of 256)
    uint64_t slot_stride;  // bytes of one ring slot
    uint64_t chan_stride;  // bytes of one channel's ring
    uint32_t R;
    uint32_t nch;
    uint32_t depth;
    uint32_t nseg;
    uint32_t nsteps;
    uint32_t inject;
#if defined(PURLIN_CHECKED)
    CheckRanges check;
#endif
    Segment seg[kSegsLarge];  // tile0 = first step of the segment
};

__device__ __forceinline__ uint64_t tag_of(uint64_t epoch, uint32_t n)
{
    return (epoch << 32) | (uint64_t)(n + 1);
}

__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* f)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint64_t* f, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_status(const int* s)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(s) : "memory");
    return v;
}

// Bounded wait of one CTA for *flag >= want.  Thread 0 polls, the first 64
// times back to back (a short message's next step is usually a round trip
// away) and then with a 100 ns sleep between polls; the outcome is shared
// through shared memory.  Returns false if the CTA must leave (this wait timed
// out, or another CTA recorded an error).
__device__ bool cta_wait(const SnacParams& p, const uint64_t* flag, uint64_t want)
{
    __shared__ int go;
    if (threadIdx.x == 0) {
        int ok = 1;
        uint64_t spins = 0, start = 0;
        while (ld_acquire(flag) < want) {
            if (ld_status(p.status) != 0) { ok = 0; break; }
            ++spins;
            if ((spins & 31) == 0) {
                uint64_t t = now_ns();
                if (start == 0) start = t;
                if (t - start > p.timeout_ns || spins > p.max_spins) {
                    atomicCAS(p.status, 0, (int)PURLIN_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
            if (spins > 64) __nanosleep(100);
        }
        go = ok;
    }
    __syncthreads();
    const bool ok = go != 0;
    __syncthreads();  // `go` is rewritten by the next wait
    return ok;
}

// Publish this CTA's work of the step: every thread's accesses happen before
// the release store of the tag.
__device__ __forceinline__ void cta_notify(uint64_t* flag, uint64_t tag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        st_release(flag, tag);
    }
}

__device__ __forceinline__ const Segment& step_segment(const SnacParams& p, uint32_t i)
{
    int lo = 0, hi = (int)p.nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile0 <= i) lo = mid;
        else hi = mid - 1;
    }
    return p.seg[lo];
}

__device__ __forceinline__ uint64_t* slot_flags(const SnacParams& p, uint32_t ch, uint32_t slot)
{
    return p.flags + ((uint64_t)ch * p.depth + slot) * kFlagsPerSlot;
}

__device__ __forceinline__ char* slot_data(const SnacParams& p, uint32_t ch, uint32_t slot)
{
    return p.staging + (uint64_t)ch * p.chan_stride + (uint64_t)slot * p.slot_stride;
}

// ------------------------------------------------------- CTA-wide data movers

// Copy len bytes src -> dst (or -> out[r] + dst_off for every r when FAN),
// in units of B bytes, four units per thread in flight.
// `skip` (an address, 0 for none): with FAN, a destination range starting there is
// the source of an in-place AllGather block and is left alone.
template <int B>
__device__ __forceinline__ void store_pol(char* d, const atom::Unit<B>& u, uint64_t pol)
{
    if constexpr (B >= 16) atom::store(d, u.v, pol);
    else atom::store_unit<B>(d, u);
}

template <int B, bool SRC_CG>
__device__ __forceinline__ void load_pol(atom::Unit<B>& u, const char* s, uint64_t pol)
{
    if constexpr (B >= 16 && !SRC_CG) atom::load(u.v, s, pol);
    else atom::load_unit<B, SRC_CG>(u, s);
}

template <int B, bool SRC_CG, bool FAN>
__device__ __forceinline__ void cta_copy(const SnacParams& p, char* dst, uint64_t dst_off,
                                         const char* src, uint64_t len, uintptr_t skip,
                                         uint64_t lpol, uint64_t spol)
{
    constexpr int U = 4;
    for (uint64_t base = 0; base < len; base += (uint64_t)kSnacThreads * B * U) {
        atom::Unit<B> u[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t o = base + (uint64_t)(k * kSnacThreads + threadIdx.x) * B;
            if (o < len) load_pol<B, SRC_CG>(u[k], src + o, lpol);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t o = base + (uint64_t)(k * kSnacThreads + threadIdx.x) * B;
            if (o >= len) continue;
            if (FAN) {
                for (int r = 0; r < (int)p.R; ++r) {
                    char* d = p.out[r] + dst_off + o;
                    if ((uintptr_t)d != skip + o) store_pol<B>(d, u[k], spol);
                }
            } else {
                store_pol<B>(dst + o, u[k], spol);
            }
        }
    }
}

// MAXU: the widest unit a launch's plan holds (5: 32 bytes; 4: 16 bytes, the
// sums of launches that hold a shifted body), so that the kernels serving
// those launches carry no 32-byte paths and keep their registers.
template <bool SRC_CG, bool FAN, int MAXU = 5>
__device__ void cta_copy_any(const SnacParams& p, int unit_log2, char* dst, uint64_t dst_off,
                             const char* src, uint64_t len, uintptr_t skip, uint64_t lpol,
                             uint64_t spol)
{
    switch (unit_log2) {
    case 5:
        if constexpr (MAXU >= 5) cta_copy<32, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol);
        break;
    case 4: cta_copy<16, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol); break;
    case 3: cta_copy<8, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol); break;
    case 2: cta_copy<4, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol); break;
    case 1: cta_copy<2, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol); break;
    default: cta_copy<1, SRC_CG, FAN>(p, dst, dst_off, src, len, skip, lpol, spol); break;
    }
}

// STAGE of a sum's step: the chunk of every source rank into its part of the
// slot.  All R loads of a unit are in flight before the first staging store,
// so one step costs about one memory round trip, not R of them.
template <int B>
__device__ __forceinline__ void cta_stage_ranks(const SnacParams& p, char* staged,
                                                uint64_t src_off, uint64_t len, uint64_t lpol)
{
    const int R = (int)p.R;
    for (uint64_t o = (uint64_t)threadIdx.x * B; o < len; o += (uint64_t)kSnacThreads * B) {
        atom::Unit<B> u[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) load_pol<B, false>(u[r], p.in[r] + src_off + o, lpol);
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) atom::store_unit<B>(staged + r * p.chunk + o, u[r]);
    }
}

template <int MAXU = 5>
__device__ void cta_stage_any(const SnacParams& p, int unit_log2, char* staged, uint64_t src_off,
                              uint64_t len, uint64_t lpol)
{
    switch (unit_log2) {
    case 5:
        if constexpr (MAXU >= 5) cta_stage_ranks<32>(p, staged, src_off, len, lpol);
        break;
    case 4: cta_stage_ranks<16>(p, staged, src_off, len, lpol); break;
    case 3: cta_stage_ranks<8>(p, staged, src_off, len, lpol); break;
    case 2: cta_stage_ranks<4>(p, staged, src_off, len, lpol); break;
    case 1: cta_stage_ranks<2>(p, staged, src_off, len, lpol); break;
    default: cta_stage_ranks<1>(p, staged, src_off, len, lpol); break;
    }
}

// Atom::reduce over the R staged pieces (stride `stride` apart) into dst.
template <typename T, int ORDER, int B>
__device__ __forceinline__ void cta_reduce_vec(const SnacParams& p, char* dst, const char* staged,
                                               uint64_t len, uint64_t spol)
{
    const int R = (int)p.R;
    for (uint64_t o = (uint64_t)threadIdx.x * B; o < len; o += (uint64_t)kSnacThreads * B) {
        atom::Vec<B> v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) atom::load_cg(v[r], staged + r * p.chunk + o);
        atom::Vec<B> out;
        atom::reduce_unit<T, ORDER, B>(v, R, out);
        atom::store(dst + o, out, spol);
    }
}

template <typename T, int ORDER>
__device__ __forceinline__ void cta_reduce_elem(const SnacParams& p, char* dst, const char* staged,
                                                uint64_t len)
{
    const int R = (int)p.R;
    for (uint64_t o = (uint64_t)threadIdx.x * T::kBytes; o < len; o += (uint64_t)kSnacThreads * T::kBytes) {
        float v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) v[r] = (r < R) ? T::load1_cg(staged + r * p.chunk + o) : 0.0f;
        T::store1(dst + o, atom::fold<ORDER>(v, R));
    }
}

template <typename T, int ORDER, int MAXU = 5>
__device__ void cta_reduce(const SnacParams& p, int unit_log2, char* dst, const char* staged,
                           uint64_t len, uint64_t spol)
{
    if (unit_log2 == 5) {
        if constexpr (MAXU >= 5) cta_reduce_vec<T, ORDER, 32>(p, dst, staged, len, spol);
    }
    else if (unit_log2 == 4) cta_reduce_vec<T, ORDER, 16>(p, dst, staged, len, spol);
    else cta_reduce_elem<T, ORDER>(p, dst, staged, len);
}

// STAGE of a reduced chunk: Atom::reduce over the sources' chunk, written to
// the slot (all R loads of a unit in flight before the fold).
template <typename T, int ORDER, int B>
__device__ __forceinline__ void cta_reduce_src_vec(const SnacParams& p, char* dst,
                                                   uint64_t src_off, uint64_t len, uint64_t lpol,
                                                   uint64_t spol)
{
    const int R = (int)p.R;
    for (uint64_t o = (uint64_t)threadIdx.x * B; o < len; o += (uint64_t)kSnacThreads * B) {
        atom::Vec<B> v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) atom::load(v[r], p.in[r] + src_off + o, lpol);
        atom::Vec<B> out;
        atom::reduce_unit<T, ORDER, B>(v, R, out);
        atom::store(dst + o, out, spol);
    }
}

template <typename T, int ORDER>
__device__ __forceinline__ void cta_reduce_src_elem(const SnacParams& p, char* dst,
                                                    uint64_t src_off, uint64_t len)
{
    const int R = (int)p.R;
    for (uint64_t o = (uint64_t)threadIdx.x * T::kBytes; o < len; o += (uint64_t)kSnacThreads * T::kBytes) {
        float v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) v[r] = (r < R) ? T::load1(p.in[r] + src_off + o) : 0.0f;
        T::store1(dst + o, atom::fold<ORDER>(v, R));
    }
}

template <typename T, int ORDER, int MAXU = 5>
__device__ void cta_reduce_src(const SnacParams& p, int unit_log2, char* dst, uint64_t src_off,
                               uint64_t len, uint64_t lpol, uint64_t spol)
{
    if (unit_log2 == 5) {
        if constexpr (MAXU >= 5) cta_reduce_src_vec<T, ORDER, 32>(p, dst, src_off, len, lpol, spol);
    }
    else if (unit_log2 == 4) cta_reduce_src_vec<T, ORDER, 16>(p, dst, src_off, len, lpol, spol);
    else cta_reduce_src_elem<T, ORDER>(p, dst, src_off, len);
}

// ------------------------------------------------ shifted bodies (producer)
// A step of a shifted body (Segment::shift != 0): the producer reads aligned
// source blocks and writes the step's units, realigned to the destinations'
// grid, into the slot, so the consumer works on aligned data.  Lanes as in the
// zero-staging kernels: a warp loads 32 blocks and writes the 31 units between
// them.  The block after a step's last unit is the next step's first (or the
// segment's last one, which holds its last bytes): within the segment.  A
// shifted step is a whole number of units.

// Copy a step's len bytes from src (any offset) to dst (unit-aligned).  The
// step's word offset is fixed at compile time (one branch per step), so a unit
// is realigned with one shuffle per word it needs from the next lane and one
// funnel shift per word; each thread has two units in flight.
template <int B>
__device__ void cta_copy_shifted(const char* src, char* dst, uint64_t len, uint64_t lpol,
                                 uint64_t spol)
{
    constexpr int W = B / 4;
    constexpr int WARPS = kSnacThreads / 32;
    constexpr int U = 2;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int shift = (int)(reinterpret_cast<uintptr_t>(src) & (B - 1));
    const uint64_t n = len / B;
    const uint64_t nblocks = shift ? n + 1 : n;
    const uint32_t bits = (uint32_t)(shift & 3) * 8;
    with_word_offset<W>(shift >> 2, [&](auto A) {
        for (uint64_t row = 0; row < n; row += (uint64_t)WARPS * 31 * U) {
            atom::Vec<B> v[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
                if (q < nblocks) {
                    atom::load(v[k], at(src, q * B, shift), lpol);
                } else {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[k].w[i] = 0u;
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
                atom::Vec<B> out;
                realign_from_next<W, decltype(A)::value>(v[k].w, bits, out.w);
                if (lane == 31 || q >= n) continue;
                atom::store(dst + q * B, out, spol);
            }
        }
    });
}

__device__ void cta_copy_shifted_any(int unit_log2, const char* src, char* dst, uint64_t len,
                                     uint64_t lpol, uint64_t spol)
{
    if (unit_log2 == 5) cta_copy_shifted<32>(src, dst, len, lpol, spol);
    else cta_copy_shifted<16>(src, dst, len, lpol, spol);
}

// Rows of a shifted step of a sum with the inputs staged, sources on one
// offset: every rank's chunk realigned into its part of the slot with the word
// offset fixed at compile time, the R ranks' blocks of kMaxRanks / NR units
// loaded before the first store (R <= NR).
template <int NR>
__device__ void stage_ranks_shifted_rows(const SnacParams& p, char* staged, uint64_t src_off,
                                         uint64_t len, uint64_t lpol)
{
    constexpr int B = 16;
    constexpr int W = B / 4;
    constexpr int WARPS = kSnacThreads / 32;
    constexpr int U = kMaxRanks / NR;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int R = (int)p.R;
    const uint64_t n = len / B;
    const int shift = (int)((reinterpret_cast<uintptr_t>(p.in[0]) + src_off) & (B - 1));
    const uint32_t bits = (uint32_t)(shift & 3) * 8;
    with_word_offset<W>(shift >> 2, [&](auto A) {
        for (uint64_t row = 0; row < n; row += (uint64_t)WARPS * 31 * U) {
            atom::Vec<B> v[U][NR];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r < R && q < n + 1) {
                        atom::load(v[k][r], at(p.in[r], src_off + q * B, shift), lpol);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[k][r].w[i] = 0u;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= R) continue;
                    atom::Vec<B> out;
                    realign_from_next<W, decltype(A)::value>(v[k][r].w, bits, out.w);
                    if (lane != 31 && q < n) atom::store(staged + r * p.chunk + q * B, out);
                }
            }
        }
    });
}

// STAGE of a shifted step of a sum with the inputs staged: every rank's chunk
// realigned into its part of the slot (16-byte units, a shifted sum's width).
// Sources on one offset: stage_ranks_shifted_rows; sources on different
// offsets: each rank's blocks realigned on their own offset.
__device__ void cta_stage_ranks_shifted(const SnacParams& p, const Segment& s, char* staged,
                                        uint64_t src_off, uint64_t len, uint64_t lpol)
{
    constexpr int B = 16;
    constexpr int W = B / 4;
    constexpr int WARPS = kSnacThreads / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int R = (int)p.R;
    const uint64_t n = len / B;
    if (!(s.shift & kShiftPerRank)) {
        if (R <= 2) stage_ranks_shifted_rows<2>(p, staged, src_off, len, lpol);
        else if (R <= 4) stage_ranks_shifted_rows<4>(p, staged, src_off, len, lpol);
        else stage_ranks_shifted_rows<kMaxRanks>(p, staged, src_off, len, lpol);
        return;
    }
    int sh[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        sh[r] = r < R ? (int)((reinterpret_cast<uintptr_t>(p.in[r]) + src_off) & (B - 1)) : 0;
    for (uint64_t row = 0; row < n; row += (uint64_t)WARPS * 31) {
        const uint64_t q = row + (uint64_t)warp * 31 + lane;
        atom::Vec<B> v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r < R && q < (sh[r] ? n + 1 : n)) {
                atom::load(v[r], at(p.in[r], src_off + q * B, sh[r]), lpol);
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i) v[r].w[i] = 0u;
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r >= R) continue;
            atom::Vec<B> next, out;
#pragma unroll
            for (int i = 0; i < W; ++i) next.w[i] = __shfl_down_sync(0xffffffffu, v[r].w[i], 1);
            if (sh[r]) realign<W>(v[r].w, next.w, sh[r], out.w);
            else out = v[r];
            if (lane != 31 && q < n) atom::store(staged + r * p.chunk + q * B, out);
        }
    }
}

// Rows of a shifted sum whose sources sit on one offset: the R ranks' aligned
// blocks are folded first (the offset is a multiple of the element size, so a
// block holds whole elements of every rank at the same positions) and the sum
// is realigned once, with the word offset fixed at compile time.  NR bounds the
// rank count (R <= NR) and each thread folds kMaxRanks / NR units at once, so a
// sum of few ranks keeps as many loads in flight as one of eight.
template <typename T, int ORDER, int NR>
__device__ void reduce_src_shifted_rows(const SnacParams& p, char* dst, uint64_t src_off,
                                        uint64_t len, uint64_t lpol, uint64_t spol)
{
    constexpr int B = 16;
    constexpr int W = B / 4;
    constexpr int WARPS = kSnacThreads / 32;
    constexpr int U = kMaxRanks / NR;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int R = (int)p.R;
    const uint64_t n = len / B;
    const int shift = (int)((reinterpret_cast<uintptr_t>(p.in[0]) + src_off) & (B - 1));
    const uint32_t bits = (uint32_t)(shift & 3) * 8;
    with_word_offset<W>(shift >> 2, [&](auto A) {
        for (uint64_t row = 0; row < n; row += (uint64_t)WARPS * 31 * U) {
            atom::Vec<B> v[U][NR];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r < R && q < n + 1) {
                        atom::load(v[k][r], at(p.in[r], src_off + q * B, shift), lpol);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[k][r].w[i] = 0u;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t q = row + (uint64_t)(k * WARPS + warp) * 31 + lane;
                atom::Vec<B> y, out;
                atom::reduce_unit<T, ORDER, B, NR>(v[k], R, y);
                realign_from_next<W, decltype(A)::value>(y.w, bits, out.w);
                if (lane == 31 || q >= n) continue;
                atom::store(dst + q * B, out, spol);
            }
        }
    });
}

// Fold a step of the R sources into dst (unit-aligned; 16-byte units, a
// shifted sum's width).  Sources on one offset: reduce_src_shifted_rows.
// Sources on different offsets: each rank's block is realigned on its own
// offset before the fold.
template <typename T, int ORDER>
__device__ void cta_reduce_src_shifted(const SnacParams& p, const Segment& s, char* dst,
                                       uint64_t src_off, uint64_t len, uint64_t lpol, uint64_t spol)
{
    constexpr int B = 16;
    constexpr int W = B / 4;
    constexpr int WARPS = kSnacThreads / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int R = (int)p.R;
    const uint64_t n = len / B;
    if (!(s.shift & kShiftPerRank)) {
        if (R <= 2) reduce_src_shifted_rows<T, ORDER, 2>(p, dst, src_off, len, lpol, spol);
        else if (R <= 4) reduce_src_shifted_rows<T, ORDER, 4>(p, dst, src_off, len, lpol, spol);
        else reduce_src_shifted_rows<T, ORDER, kMaxRanks>(p, dst, src_off, len, lpol, spol);
        return;
    }
    int sh[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        sh[r] = r < R ? (int)((reinterpret_cast<uintptr_t>(p.in[r]) + src_off) & (B - 1)) : 0;
    for (uint64_t row = 0; row < n; row += (uint64_t)WARPS * 31) {
        const uint64_t q = row + (uint64_t)warp * 31 + lane;
        atom::Vec<B> v[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r < R && q < (sh[r] ? n + 1 : n)) {
                atom::load(v[r], at(p.in[r], src_off + q * B, sh[r]), lpol);
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i) v[r].w[i] = 0u;
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r >= R || sh[r] == 0) continue;
            atom::Vec<B> next;
#pragma unroll
            for (int i = 0; i < W; ++i) next.w[i] = __shfl_down_sync(0xffffffffu, v[r].w[i], 1);
            realign<W>(v[r].w, next.w, sh[r], v[r].w);
        }
        if (lane == 31 || q >= n) continue;
        atom::Vec<B> out;
        atom::reduce_unit<T, ORDER, B>(v, R, out);
        atom::store(dst + q * B, out, spol);
    }
}

// ------------------------------------------------------------------ roles

// Relaxed access to a flag-area word that a release / acquire pair orders.
__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* w)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(w) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* w, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(w), "l"(v) : "memory");
}

// Every kind hands out steps from a counter instead of dealing them
// round-robin: a channel whose SM drains faster takes more steps, so the
// slowest SMs do not set the time.  The producer records the step in the slot's step
// word before notifying; the consumer reads it after the acquire.  When the plan
// has one step per channel (nsteps == nch: channel ch's step is ch, and the
// counter has nothing left), every role leaves after that step instead of
// passing an end-of-steps marker down the pipeline.
template <typename T, int ORDER, int KIND, bool SHIFTED>
__device__ void producer_dynamic(const SnacParams& p, uint32_t ch, uint64_t epoch)
{
    constexpr int MAXU = snac_max_unit(KIND, SHIFTED);
    __shared__ uint64_t step_s;
    const uint64_t lpol = atom::l2_policy(kL2EvictFirst);
    const uint64_t spol = atom::l2_policy(kL2Normal);
    // A channel's first step is its own index (steps >= channels); every later
    // one comes from the counter when the channel is ready for it (taking it
    // one step ahead, to hide the atomic's round trip, balanced worse:
    // AllReduce 192.5 -> 201.2 us).
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % p.depth;
        uint64_t* f = slot_flags(p, ch, slot);
        if (n >= p.depth && !cta_wait(p, f + kFree, tag_of(epoch, n - p.depth))) return;
        if (threadIdx.x == 0)
            step_s = n == 0 ? (uint64_t)ch : (uint64_t)p.nch + atomicAdd(p.step_word, 1ull);
        __syncthreads();
        const uint64_t i = step_s;
        __syncthreads();  // step_s is rewritten next step
        if (i >= p.nsteps) {
            if (threadIdx.x == 0) st_relaxed(f + kStepOf, kNoStep);
            cta_notify(f + kReady, tag_of(epoch, n));
            return;
        }
        const Segment& s = step_segment(p, (uint32_t)i);
        const uint64_t off = (uint64_t)((uint32_t)i - s.tile0) * p.chunk;
        const uint64_t len = min(p.chunk, s.bytes - off);
        bool staged = false;
        if constexpr (SHIFTED) {
            if (s.shift) {
                // realigned to the destinations' grid while staged
                char* slot_p = slot_data(p, ch, slot);
                if (KIND == kRSY || KIND == kARY) {
                    cta_reduce_src_shifted<T, ORDER>(p, s, slot_p, s.src_off + off, len, lpol,
                                                     spol);
                } else if (KIND == kRS || KIND == kAR) {
                    cta_stage_ranks_shifted(p, s, slot_p, s.src_off + off, len, lpol);
                } else {
                    cta_copy_shifted_any(s.unit_log2, p.in[s.src] + s.src_off + off, slot_p, len,
                                         lpol, spol);
                }
                staged = true;
            }
        }
        if (!staged) {
            if (KIND == kRSY || KIND == kARY) {
                cta_reduce_src<T, ORDER, MAXU>(p, s.unit_log2, slot_data(p, ch, slot), s.src_off + off,
                                         len, lpol, spol);
            } else if (KIND == kRS || KIND == kAR) {
                cta_stage_any<MAXU>(p, s.unit_log2, slot_data(p, ch, slot), s.src_off + off, len,
                                    lpol);
            } else {
                cta_copy_any<false, false>(p, s.unit_log2, slot_data(p, ch, slot), 0,
                                           p.in[s.src] + s.src_off + off, len, 0, lpol, spol);
            }
        }
        if (threadIdx.x == 0) st_relaxed(f + kStepOf, i);
        if (p.inject && ch == 0 && n == 0) continue;  // testing: this notify never happens
        cta_notify(f + kReady, tag_of(epoch, n));
        if (p.nsteps == p.nch) return;  // one step per channel: no end-of-steps round
    }
}

template <typename T, int ORDER, int KIND, int MAXU>
__device__ void consumer_dynamic(const SnacParams& p, uint32_t ch, uint64_t epoch)
{
    __shared__ uint64_t step_s;
    // AllReduce, AllGather and AllToAll outputs are written once: evict-first.
    // A ReduceScatter's stay at normal priority (a following AllGather reads
    // them).
    const uint64_t lpol = atom::l2_policy(kL2Normal);
    const uint64_t spol =
        atom::l2_policy((KIND == kRSY || KIND == kRS) ? kL2Normal : kL2EvictFirst);
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % p.depth;
        uint64_t* f = slot_flags(p, ch, slot);
        if (!cta_wait(p, f + kReady, tag_of(epoch, n))) return;
        if (threadIdx.x == 0) step_s = ld_relaxed(f + kStepOf);
        __syncthreads();
        const uint64_t i = step_s;
        __syncthreads();
        if (i >= p.nsteps) return;  // kNoStep: the producer is done
        const Segment& s = step_segment(p, (uint32_t)i);
        const uint64_t off = (uint64_t)((uint32_t)i - s.tile0) * p.chunk;
        const uint64_t len = min(p.chunk, s.bytes - off);
        const char* staged = slot_data(p, ch, slot);
        if (KIND == kRS) {
            cta_reduce<T, ORDER, MAXU>(p, s.unit_log2, p.out[s.dst] + s.dst_off + off, staged, len,
                                 spol);
        } else if (KIND == kARY) {
            // In-place AllReduce (out[r] == in[r]): this step's input range was
            // read by the producer before the ready tag was published.
            cta_copy_any<true, true, MAXU>(p, s.unit_log2, nullptr, s.dst_off + off, staged, len,
                                           0, lpol, spol);
        } else if (KIND == kAG) {
            cta_copy_any<true, true, MAXU>(p, s.unit_log2, nullptr, s.dst_off + off, staged, len,
                                     (uintptr_t)(p.in[s.src] + s.src_off + off), lpol, spol);
        } else {
            cta_copy_any<true, false, MAXU>(p, s.unit_log2, p.out[s.dst] + s.dst_off + off, 0, staged,
                                      len, 0, lpol, spol);
        }
        cta_notify(f + kFree, tag_of(epoch, n));
        if (p.nsteps == p.nch) return;
    }
}

// The three-role AllReduce (the R input chunks staged): the consumer sums them
// into the slot's y part and records the step there; the gatherer copies y to
// all R outputs.
template <typename T, int ORDER, int MAXU>
__device__ void consumer_ar(const SnacParams& p, uint32_t ch, uint64_t epoch)
{
    __shared__ uint64_t step_s;
    // The consumer writes into the ring's y part, which the gatherer reads.
    const uint64_t spol = atom::l2_policy(kL2Normal);
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % p.depth;
        uint64_t* f = slot_flags(p, ch, slot);
        if (!cta_wait(p, f + kReady, tag_of(epoch, n))) return;
        if (threadIdx.x == 0) step_s = ld_relaxed(f + kStepOf);
        __syncthreads();
        const uint64_t i = step_s;
        __syncthreads();
        // the y part of this slot is free once the gatherer is done with step n - depth
        if (n >= p.depth && !cta_wait(p, f + kYFree, tag_of(epoch, n - p.depth))) return;
        if (i < p.nsteps) {
            const Segment& s = step_segment(p, (uint32_t)i);
            const uint64_t off = (uint64_t)((uint32_t)i - s.tile0) * p.chunk;
            const uint64_t len = min(p.chunk, s.bytes - off);
            char* staged = slot_data(p, ch, slot);
            cta_reduce<T, ORDER, MAXU>(p, s.unit_log2, staged + (uint64_t)p.R * p.chunk, staged, len,
                                 spol);
        }
        if (threadIdx.x == 0) st_relaxed(f + kYStepOf, i);  // kNoStep passes through
        cta_notify(f + kFree, tag_of(epoch, n));
        if (threadIdx.x == 0) st_release(f + kYReady, tag_of(epoch, n));
        if (i >= p.nsteps || p.nsteps == p.nch) return;
    }
}

template <int MAXU>
__device__ void gatherer(const SnacParams& p, uint32_t ch, uint64_t epoch)
{
    __shared__ uint64_t step_s;
    // The R outputs are written once: evict-first keeps the ring in L2.
    const uint64_t lpol = atom::l2_policy(kL2Normal);
    const uint64_t spol = atom::l2_policy(kL2EvictFirst);
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % p.depth;
        uint64_t* f = slot_flags(p, ch, slot);
        if (!cta_wait(p, f + kYReady, tag_of(epoch, n))) return;
        if (threadIdx.x == 0) step_s = ld_relaxed(f + kYStepOf);
        __syncthreads();
        const uint64_t i = step_s;
        __syncthreads();
        if (i >= p.nsteps) return;
        const Segment& s = step_segment(p, (uint32_t)i);
        const uint64_t off = (uint64_t)((uint32_t)i - s.tile0) * p.chunk;
        const uint64_t len = min(p.chunk, s.bytes - off);
        const char* y = slot_data(p, ch, slot) + (uint64_t)p.R * p.chunk;
        // In-place AllReduce writes out[r] == in[r]; this step's input range
        // was staged before the y tag was published, so the writes are safe.
        cta_copy_any<true, true, MAXU>(p, s.unit_log2, nullptr, s.dst_off + off, y, len, 0, lpol,
                                       spol);
        cta_notify(f + kYFree, tag_of(epoch, n));
        if (p.nsteps == p.nch) return;
    }
}

// SHIFTED: the plan holds a shifted body (only such launches carry that path).
template <typename T, int ORDER, int KIND, bool SHIFTED>
__global__ void __launch_bounds__(kSnacThreads, kSnacCtasPerSm) snac_kernel(const __grid_constant__ SnacParams p)
{
    PURLIN_CHECK_BEGIN(p);
    __shared__ uint64_t epoch_s;
    if (threadIdx.x == 0) {
        uint64_t prev;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(prev) : "l"(p.epoch_word) : "memory");
        epoch_s = prev + 1;
    }
    __syncthreads();
    const uint64_t epoch = epoch_s;
    constexpr int MAXU = snac_max_unit(KIND, SHIFTED);
    const uint32_t role = blockIdx.x / p.nch;
    const uint32_t ch = blockIdx.x % p.nch;
    if (role == 0) {
        producer_dynamic<T, ORDER, KIND, SHIFTED>(p, ch, epoch);
    } else if constexpr (KIND == kAR) {
        if (role == 1) consumer_ar<T, ORDER, MAXU>(p, ch, epoch);
        else gatherer<MAXU>(p, ch, epoch);
    } else {
        consumer_dynamic<T, ORDER, KIND, MAXU>(p, ch, epoch);
    }
    // Whatever path a role left by (done, or an error seen), the last CTA to
    // get here publishes the epoch for the next call and resets the counter.
    // No CTA reads the epoch word after its start, and every CTA has started
    // before the last one arrives, so all of them used the same epoch.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.done_word, 1u) == gridDim.x - 1) {
            atomicExch(p.done_word, 0u);
            atomicExch(p.step_word, 0ull);
            __threadfence();
            st_release(p.epoch_word, epoch);
        }
    }
}

using SnacKernel = void (*)(SnacParams);

template <typename T, int KIND, bool SH>
SnacKernel pick_order(int order)
{
    return order == 0 ? snac_kernel<T, 0, KIND, SH> : snac_kernel<T, 1, KIND, SH>;
}

template <int KIND, bool SH>
SnacKernel pick_dtype(int dtype, int order)
{
    if (dtype == kF32) return pick_order<atom::F32, KIND, SH>(order);
    if (dtype == kBF16) return pick_order<atom::BF16, KIND, SH>(order);
    return pick_order<atom::F16, KIND, SH>(order);
}

template <bool SH>
SnacKernel kernel_for_sh(Coll coll, int dtype, int order, bool stage_y)
{
    switch (coll) {
    case Coll::ReduceScatter:
        return stage_y ? pick_dtype<kRSY, SH>(dtype, order) : pick_dtype<kRS, SH>(dtype, order);
    case Coll::AllReduce:
        return stage_y ? pick_dtype<kARY, SH>(dtype, order) : pick_dtype<kAR, SH>(dtype, order);
    case Coll::AllGather: return snac_kernel<atom::F32, 0, kAG, SH>;
    default: return snac_kernel<atom::F32, 0, kA2A, SH>;
    }
}

SnacKernel kernel_for(Coll coll, int dtype, int order, bool stage_y, bool shifted)
{
    return shifted ? kernel_for_sh<true>(coll, dtype, order, stage_y)
                   : kernel_for_sh<false>(coll, dtype, order, stage_y);
}

int roles_of(Coll coll, bool stage_y) { return coll == Coll::AllReduce && !stage_y ? 3 : 2; }

// Widest access of the staged kernels (tuning knob for measurements only).
int snac_unit_log2()
{
    static const int u = [] {
        const char* e = std::getenv("PURLIN_SNAC_UNIT");
        return (e && std::atoi(e) == 16) ? 4 : 5;
    }();
    return u;
}

int sub_slots(Coll coll, int R, bool stage_y)
{
    if (stage_y) return 1;
    if (coll == Coll::AllReduce) return R + 1;
    if (coll == Coll::ReduceScatter) return R;
    return 1;
}

}  // namespace

purlin_status_t snac_geometry(int R, Coll coll, bool stage_y, const SnacConfig& cfg,
                              int resident_per_sm, uint64_t total_bytes, size_t* chunk_out,
                              int* depth_out, int* channels_out)
{
    const long resident_channels = (long)resident_per_sm * cfg.sms / roles_of(coll, stage_y);
    size_t chunk = cfg.chunk_bytes;
    if (!chunk) {
        // the measured default, but small enough that a short message still
        // spreads over every channel the GPU can hold (at least 1 KiB)
        const long target = std::max<long>(1, std::min<long>(resident_channels, kMaxChannels));
        const uint64_t spread = (total_bytes + (uint64_t)target - 1) / (uint64_t)target;
        chunk = std::min<size_t>(default_chunk(coll, R, stage_y),
                                 std::max<size_t>(kMinAutoChunk, (size_t)spread));
    }
    chunk = std::max<size_t>(256, (chunk + 255) & ~(size_t)255);
    const int depth = cfg.depth ? cfg.depth : kDefaultDepth;
    const size_t slot = (size_t)sub_slots(coll, R, stage_y) * chunk;
    const size_t ring = (size_t)depth * slot;
    const long by_ring = ring ? (long)(cfg.staging_bytes / ring) : 0;
    // the last three flag words hold the epoch, the completion counter and
    // the step counter
    const long by_flags = (long)((cfg.flag_words - 3) / ((size_t)depth * kFlagsPerSlot));
    const long by_residency = resident_channels;
    long nch = cfg.channels ? cfg.channels : kMaxChannels;
    nch = std::min({nch, by_ring, by_flags, by_residency});
    if (nch < 1) return PURLIN_ERR_UNSUPPORTED;  // ring too small for this chunk/depth
    *chunk_out = chunk;
    *depth_out = depth;
    *channels_out = (int)nch;
    return PURLIN_OK;
}

namespace {

static_assert(sizeof(SnacParams) <= kMaxLaunchParams, "launch parameter block");

// Plan one staged call into k: the kernel, its launch shape and its parameter
// block (k.grid = 0: nothing to launch).
purlin_status_t plan_into(KernelLaunch& k, const SnacRequest& rq, const SnacConfig& cfg,
                          SnacLaunch* launch)
{
    SnacParams& p = *reinterpret_cast<SnacParams*>(k.params);
    std::memset(&p, 0, sizeof(p));
    k.grid = 0;
    const bool reduce = rq.coll == Coll::ReduceScatter || rq.coll == Coll::AllReduce;
    uint32_t ntiles = 0;
    // shifted bodies: the producer realigns them while staging
    const bool allow_shift = true;
    int nseg = layout_segments(rq.pieces, rq.npieces, rq.R, rq.in, rq.out, rq.esz, reduce,
                               reduce ? kTileUnitsReduce : kTileUnitsCopy, snac_unit_log2(),
                               allow_shift, p.seg, kSegsLarge, &ntiles);
    if (nseg < 0) return PURLIN_ERR_UNSUPPORTED;
    bool shifted = false;
    for (int i = 0; i < nseg; ++i) shifted |= p.seg[i].shift != 0;
    if (shifted && reduce && snac_unit_log2() > 4) {
        // the kernels serving shifted sums take 16-byte vector bodies only
        nseg = layout_segments(rq.pieces, rq.npieces, rq.R, rq.in, rq.out, rq.esz, reduce,
                               kTileUnitsReduce, 4, allow_shift, p.seg, kSegsLarge, &ntiles);
        if (nseg < 0) return PURLIN_ERR_UNSUPPORTED;
    }

    SnacKernel kernel = kernel_for(rq.coll, rq.dtype, rq.order, rq.stage_y, shifted);
    const int resident = resident_ctas_of(reinterpret_cast<const void*>(kernel), kSnacThreads);
    if (resident < 1) return PURLIN_ERR_CUDA;
    size_t chunk = 0;
    int depth = 0, nch = 0;
    uint64_t total_bytes = 0;
    for (int i = 0; i < nseg; ++i) total_bytes += p.seg[i].bytes;
    purlin_status_t st = snac_geometry(rq.R, rq.coll, rq.stage_y, cfg, resident, total_bytes,
                                       &chunk, &depth, &nch);
    if (st != PURLIN_OK) return st;

    // Steps: every segment cut into chunks of `chunk` bytes.
    uint64_t steps = 0;
    for (int i = 0; i < nseg; ++i) {
        p.seg[i].tile0 = (uint32_t)steps;
        steps += (p.seg[i].bytes + chunk - 1) / chunk;
        if (steps > 0xffffffffull) return PURLIN_ERR_UNSUPPORTED;
    }
    if (steps == 0) {
        *launch = SnacLaunch{0, 0, kSnacThreads, depth, 0, chunk};
        return PURLIN_OK;
    }
    nch = (int)std::min<uint64_t>((uint64_t)nch, steps);

    for (int r = 0; r < rq.R; ++r) {
        p.in[r] = reinterpret_cast<const char*>(rq.in[r]);
        p.out[r] = reinterpret_cast<char*>(rq.out[r]);
    }
    p.staging = cfg.staging;
    p.flags = cfg.flags;
    p.status = cfg.status;
    p.epoch_word = cfg.flags + cfg.flag_words - 1;
    p.done_word = reinterpret_cast<uint32_t*>(cfg.flags + cfg.flag_words - 2);
    p.step_word = reinterpret_cast<unsigned long long*>(cfg.flags + cfg.flag_words - 3);
    p.timeout_ns = cfg.timeout_ns;
    p.max_spins = cfg.timeout_ns / 64 + 65536;
    p.chunk = chunk;
    p.slot_stride = (uint64_t)sub_slots(rq.coll, rq.R, rq.stage_y) * chunk;
    p.chan_stride = (uint64_t)depth * p.slot_stride;
    p.R = (uint32_t)rq.R;
    p.nch = (uint32_t)nch;
    p.depth = (uint32_t)depth;
    p.nseg = (uint32_t)nseg;
    p.nsteps = (uint32_t)steps;
    p.inject = (uint32_t)cfg.inject_skip_notify;
#if defined(PURLIN_CHECKED)
    // the call's buffers and the staging ring
    if (rq.check) p.check = *rq.check;
    add_range(p.check, reinterpret_cast<uint64_t>(cfg.staging), cfg.staging_bytes);
#endif

    const int grid = nch * roles_of(rq.coll, rq.stage_y);
    k.func = reinterpret_cast<const void*>(kernel);
    k.grid = (unsigned)grid;
    k.block = kSnacThreads;
    k.smem = 0;
    k.pdl = false;
    k.cooperative = true;  // every waiter's partner must be resident
    k.params_bytes = sizeof(SnacParams);
    *launch = SnacLaunch{1, grid, kSnacThreads, depth, nch, chunk};
    return PURLIN_OK;
}

}  // namespace

purlin_status_t snac_plan(const SnacRequest& rq, const SnacConfig& cfg, KernelLaunch& k,
                          SnacLaunch* launch)
{
    return plan_into(k, rq, cfg, launch);
}

purlin_status_t snac_run_on_stack(const SnacRequest& rq, const SnacConfig& cfg,
                                  cudaStream_t stream, SnacLaunch* launch)
{
    KernelLaunch k;
    purlin_status_t st = plan_into(k, rq, cfg, launch);
    if (st != PURLIN_OK || k.grid == 0) return st;
    return launch_kernel(k, stream) == cudaSuccess ? PURLIN_OK : PURLIN_ERR_CUDA;
}

}  // namespace purlin
