// zs_kernels.cuh -- zero-staging ("ZS") Atom kernels for sm_103a (device code;
// their host-side selection and launch are in zs_kernels.cu).
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives",
// Figure 10: "Purlin-ZS omits staging" when buffers are directly accessible.  On
// one GPU every virtual rank's buffer is directly accessible, so the ZS kernels
// read the sources and write the destinations in one pass:
//   - zs_reduce: ReduceScatter(V) (one destination per segment) and the fused
//     AllReduce of Figure 6 (each summed unit written to all R outputs);
//   - zs_copy:   AllGather(V) (each unit written to all R outputs) and
//     AllToAll(V) (one destination per segment).
// Work is a flat space of tiles (plan.h) walked grid-stride; the host sizes the
// grid (capi.cpp: several waves of CTAs, at most one per tile).  Each CTA finds
// a tile's segment by binary search over the segments' first tiles, which sit
// in the kernel's constant parameter bank.
#pragma once

#include <type_traits>

#include "atom.cuh"
#include "internal.h"
#include "purlin.h"

namespace purlin {

namespace {

template <int MAXSEG>
__device__ __forceinline__ const Segment& segment_of(const ZsParams<MAXSEG>& p, uint32_t t)
{
    int lo = 0, hi = (int)p.nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile0 <= t) lo = mid;
        else hi = mid - 1;
    }
    return p.seg[lo];
}

// Programmatic dependent launch: the grid may have been scheduled before the
// previous kernel on the stream finished; griddepcontrol.wait blocks until that
// kernel has completed and its writes are visible (it returns at once when the
// launch had no programmatic dependency).  Triggering dependents right after
// lets the next collective's CTAs be scheduled while this one runs.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ shifted bodies
// A shifted segment (Segment::shift != 0) has its destinations aligned to its
// unit of BYTES while its sources start `shift` bytes past a unit boundary (a
// V-collective whose partition offsets are not multiples of the vector).
// Lane l of a warp loads the aligned source block q + l -- for a sum on one
// offset, the R ranks' blocks folded first: `shift` is a multiple of the
// element size, so the realignment moves whole elements -- and destination unit
// q + l is that block's last BYTES - shift bytes followed by the first `shift`
// bytes of the next block, which lane l + 1 holds.  (A sum whose ranks sit on
// different offsets, kShiftPerRank, realigns each rank's block the same way
// before the fold.)  Each warp's 32 lanes thus write 31 units (lane 31 only
// lends its block); every block loaded holds a byte of the segment, so no load
// leaves the pages the segment lies in.

// out = (lo ++ hi)[shift, shift + 4W) as bytes, 0 < shift < 4W, with no
// dynamically indexed registers: a log-depth word rotation, then a funnel
// shift for the bytes within a word.
template <int W>
__device__ __forceinline__ void realign(const uint32_t (&lo)[W], const uint32_t (&hi)[W],
                                        int shift, uint32_t (&out)[W])
{
    uint32_t c[2 * W];
#pragma unroll
    for (int i = 0; i < W; ++i) {
        c[i] = lo[i];
        c[W + i] = hi[i];
    }
    const int words = shift >> 2;
#pragma unroll
    for (int k = W / 2; k >= 1; k >>= 1) {
        const bool take = (words & k) != 0;
#pragma unroll
        for (int i = 0; i + k < 2 * W; ++i) c[i] = take ? c[i + k] : c[i];
    }
    const uint32_t bits = (uint32_t)(shift & 3) * 8;
#pragma unroll
    for (int j = 0; j < W; ++j) out[j] = __funnelshift_r(c[j], c[j + 1], bits);
}

// Calls f(std::integral_constant<int, a>) for a runtime word offset a in
// [0, W): a segment's shift is uniform, so the realignment below is compiled
// once per word offset and a tile branches once.
template <int W, typename F>
__device__ __forceinline__ void with_word_offset(int a, F&& f)
{
    switch (a) {
    case 0: f(std::integral_constant<int, 0>{}); break;
    case 1: f(std::integral_constant<int, 1>{}); break;
    case 2: f(std::integral_constant<int, 2>{}); break;
    case 3: f(std::integral_constant<int, 3>{}); break;
    default:
        if constexpr (W > 4) {
            switch (a) {
            case 4: f(std::integral_constant<int, 4>{}); break;
            case 5: f(std::integral_constant<int, 5>{}); break;
            case 6: f(std::integral_constant<int, 6>{}); break;
            default: f(std::integral_constant<int, 7>{}); break;
            }
        }
        break;
    }
}

// realign() for a word offset A known at compile time: the neighbour lane's
// words 0..A by shuffle (every lane calls this), then one funnel shift per
// output word.  Returns in out the unit (lo ++ next)[4A + bytes, ...).
template <int W, int A>
__device__ __forceinline__ void realign_from_next(const uint32_t (&lo)[W], uint32_t bits,
                                                  uint32_t (&out)[W])
{
    uint32_t next[A + 1];
#pragma unroll
    for (int i = 0; i <= A; ++i) next[i] = __shfl_down_sync(0xffffffffu, lo[i], 1);
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const uint32_t a = (A + j < W) ? lo[A + j] : next[A + j - W];
        const uint32_t b = (A + j + 1 < W) ? lo[A + j + 1] : next[A + j + 1 - W];
        out[j] = __funnelshift_r(a, b, bits);
    }
}

__device__ __forceinline__ const char* at(const char* base, uint64_t off, int back)
{
    return reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(base) + off - (uint64_t)back);
}

// One tile of a 16- or 32-byte vector body in a launch that holds a shifted
// sum: U = kMaxRanks / NR rows of warp runs, 31 units a warp for a shifted
// body, 32 for an aligned one (no exchange between lanes).  PER_RANK: the
// launch holds a body whose ranks' sources sit on different offsets; each
// rank's offset is then read from its address and its blocks realigned before
// the fold (a body on one offset folds first and realigns the sum once).
template <typename T, int ORDER, bool FAN_ALL, int BYTES, int NR, int THREADS, bool PER_RANK>
__device__ __forceinline__ void reduce_rows(const ZsParams<kSegsSmall>& p, const Segment& s,
                                            uint32_t tile, int R, uint64_t lpol, uint64_t spol)
{
    constexpr int U = kMaxRanks / NR;
    constexpr int W = BYTES / 4;
    constexpr int WARPS = THREADS / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool shifted = s.shift != 0;
    const int per_warp = shifted ? 31 : 32;
    const uint64_t nunits = s.bytes / BYTES;
    const uint64_t q0 =
        (uint64_t)tile * (shifted ? shifted_tile_units(THREADS * U) : THREADS * U);
    atom::Vec<BYTES> v[U][NR];
    if constexpr (!PER_RANK) {
        const int shift = s.shift;
        // a shifted body also reads the block after its last unit
        const uint64_t nblocks = shifted ? nunits + 1 : nunits;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * per_warp + lane;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < R && q < nblocks) {
                    atom::load(v[k][r], at(p.in[r], s.src_off + q * BYTES, shift), lpol);
                } else {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[k][r].w[i] = 0u;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * per_warp + lane;
            atom::Vec<BYTES> y, out;
            atom::reduce_unit<T, ORDER, BYTES, NR>(v[k], R, y);
            if (shifted) {
                atom::Vec<BYTES> next;
#pragma unroll
                for (int i = 0; i < W; ++i) next.w[i] = __shfl_down_sync(0xffffffffu, y.w[i], 1);
                if (lane == 31 || q >= nunits) continue;
                realign<W>(y.w, next.w, shift, out.w);
            } else {
                if (q >= nunits) continue;
                out = y;
            }
            const uint64_t o = s.dst_off + q * BYTES;
            if (FAN_ALL) {
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    if (r < R) atom::store(p.out[r] + o, out, spol);
            } else {
                atom::store(p.out[s.dst] + o, out, spol);
            }
        }
    } else {
        // Each rank's offset from the destinations' grid (0 on an aligned
        // body).  A rank off the grid also reads the block after the body's
        // last unit (it holds the body's last bytes); one on the grid stops at
        // the last unit.
        int sh[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r)
            sh[r] = (shifted && r < R)
                        ? (int)((reinterpret_cast<uintptr_t>(p.in[r]) + s.src_off) & (BYTES - 1))
                        : 0;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * per_warp + lane;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < R && q < (sh[r] ? nunits + 1 : nunits)) {
                    atom::load(v[k][r], at(p.in[r], s.src_off + q * BYTES, sh[r]), lpol);
                } else {
#pragma unroll
                    for (int i = 0; i < W; ++i) v[k][r].w[i] = 0u;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * per_warp + lane;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= R || sh[r] == 0) continue;
                atom::Vec<BYTES> next;
#pragma unroll
                for (int i = 0; i < W; ++i)
                    next.w[i] = __shfl_down_sync(0xffffffffu, v[k][r].w[i], 1);
                realign<W>(v[k][r].w, next.w, sh[r], v[k][r].w);
            }
            if ((shifted && lane == 31) || q >= nunits) continue;
            atom::Vec<BYTES> out;
            atom::reduce_unit<T, ORDER, BYTES, NR>(v[k], R, out);
            const uint64_t o = s.dst_off + q * BYTES;
            if (FAN_ALL) {
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    if (r < R) atom::store(p.out[r] + o, out, spol);
            } else {
                atom::store(p.out[s.dst] + o, out, spol);
            }
        }
    }
}

// One tile of a shifted copy: UNROLL rows of 31-unit warp runs.
template <int BYTES, bool FAN_ALL, int THREADS, int UNROLL, int MAXSEG>
__device__ __forceinline__ void copy_shifted(const ZsParams<MAXSEG>& p, const Segment& s,
                                          uint32_t tile, uint64_t lpol, uint64_t spol)
{
    constexpr int W = BYTES / 4;
    constexpr int WARPS = THREADS / 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int shift = s.shift;
    const uint64_t nunits = s.bytes / BYTES;
    const uint64_t q0 = (uint64_t)tile * shifted_tile_units(THREADS * UNROLL);
    atom::Vec<BYTES> v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
        const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * 31 + lane;
        if (q <= nunits) {
            atom::load(v[k], at(p.in[s.src], s.src_off + q * BYTES, shift), lpol);
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i) v[k].w[i] = 0u;
        }
    }
    const uint32_t bits = (uint32_t)(shift & 3) * 8;
    with_word_offset<W>(shift >> 2, [&](auto A) {
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
            const uint64_t q = q0 + (uint64_t)(k * WARPS + warp) * 31 + lane;
            atom::Vec<BYTES> out;
            realign_from_next<W, decltype(A)::value>(v[k].w, bits, out.w);
            if (lane == 31 || q >= nunits) continue;
            const uint64_t o = s.dst_off + q * BYTES;
            if (FAN_ALL) {
                for (int r = 0; r < (int)p.R; ++r) atom::store(p.out[r] + o, out, spol);
            } else {
                atom::store(p.out[s.dst] + o, out, spol);
            }
        }
    });
}

// ------------------------------------------------------------------ reduce

// One unit per thread (sums of more than 4 ranks, and the pairwise order).
template <typename T, int ORDER, bool FAN_ALL, int BYTES>
__device__ __forceinline__ void reduce_vector(const ZsParams<kSegsSmall>& p, const Segment& s,
                                              uint64_t off, int R, uint64_t lpol, uint64_t spol)
{
    atom::Vec<BYTES> v[kMaxRanks];
    // All R loads are issued before the first add: R independent requests in
    // flight per thread.
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        if (r < R) atom::load(v[r], p.in[r] + s.src_off + off, lpol);
    atom::Vec<BYTES> o;
    atom::reduce_unit<T, ORDER, BYTES>(v, R, o);
    if (FAN_ALL) {
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) atom::store(p.out[r] + s.dst_off + off, o, spol);
    } else {
        atom::store(p.out[s.dst] + s.dst_off + off, o, spol);
    }
}

// Several units per thread (sums of 2 to 4 ranks): U = kMaxRanks / NR of them
// for at most NR ranks (R <= NR), each warp access contiguous.  All R x U loads
// are issued before the first add, so a small rank count keeps as many
// independent requests in flight per thread as kMaxRanks ranks do.
template <typename T, int ORDER, bool FAN_ALL, int BYTES, int NR, int THREADS>
__device__ __forceinline__ void reduce_tile(const ZsParams<kSegsSmall>& p, const Segment& s,
                                            uint64_t base, int R, uint64_t lpol, uint64_t spol)
{
    constexpr int U = kMaxRanks / NR;
    const uint64_t rem = s.bytes - base;
    atom::Vec<BYTES> v[U][NR];
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const uint64_t o = (uint64_t)(k * THREADS + threadIdx.x) * BYTES;
        if (o < rem) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
                if (r < R) atom::load(v[k][r], p.in[r] + s.src_off + base + o, lpol);
        }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const uint64_t o = (uint64_t)(k * THREADS + threadIdx.x) * BYTES;
        if (o >= rem) continue;
        atom::Vec<BYTES> out;
        atom::reduce_unit<T, ORDER, BYTES, NR>(v[k], R, out);
        if (FAN_ALL) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
                if (r < R) atom::store(p.out[r] + s.dst_off + base + o, out, spol);
        } else {
            atom::store(p.out[s.dst] + s.dst_off + base + o, out, spol);
        }
    }
}

template <typename T, int ORDER, bool FAN_ALL>
__device__ __forceinline__ void reduce_element(const ZsParams<kSegsSmall>& p, const Segment& s,
                                               uint64_t off, int R)
{
    float v[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r) v[r] = (r < R) ? T::load1(p.in[r] + s.src_off + off) : 0.0f;
    float acc = atom::fold<ORDER>(v, R);
    if (FAN_ALL) {
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r)
            if (r < R) T::store1(p.out[r] + s.dst_off + off, acc);
    } else {
        T::store1(p.out[s.dst] + s.dst_off + off, acc);
    }
}

// THREADS threads per CTA: kThreads for large messages, one warp
// (kSmallThreads) for small ones.  NR bounds the rank count (R <= NR); a tile
// holds THREADS x (kMaxRanks / NR) units, so sums of 2 or 4 ranks take 4 or 2
// units per thread.  SHIFTED kernels (1: sources on one offset; 2: ranks'
// sources on different offsets) also serve shifted segments; a launch with
// none runs the kernel without that path.
template <typename T, int ORDER, bool FAN_ALL, int THREADS, int NR, int SHIFTED>
__global__ void __launch_bounds__(THREADS, THREADS == kThreads ? 2 : 16)
zs_reduce_kernel(const __grid_constant__ ZsParams<kSegsSmall> p)
{
    constexpr int U = kMaxRanks / NR;
    pdl_enter();
    PURLIN_CHECK_BEGIN(p);
    const int R = (int)p.R;
    const uint64_t lpol = atom::l2_policy(p.l2_load);
    const uint64_t spol = atom::l2_policy(p.l2_store);
    for (uint32_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const Segment& s = segment_of(p, t);
        const int ul = s.unit_log2;
        if constexpr (SHIFTED != 0) {
            // a launch holding a shifted sum is planned with 16-byte vector
            // bodies only (and element heads and tails)
            if (ul == 4) {
                reduce_rows<T, ORDER, FAN_ALL, 16, NR, THREADS, SHIFTED == 2>(p, s, t - s.tile0, R,
                                                                             lpol, spol);
            } else if (ul < 4) {
                const uint64_t base = (uint64_t)(t - s.tile0) * tile_bytes(ul, THREADS * U);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const uint64_t off = base + ((uint64_t)(k * THREADS + threadIdx.x) << ul);
                    if (off < s.bytes) reduce_element<T, ORDER, FAN_ALL>(p, s, off, R);
                }
            } else if (threadIdx.x == 0) {
                atomicCAS(p.status, 0, (int)PURLIN_ERR_UNSUPPORTED);  // not planned this way
            }
            continue;
        }
        if constexpr (U == 1) {
            // kept in this form: the one-unit kernels scheduled from the
            // general tile loop below ran up to 8 % slower (fp32 AllReduce)
            const uint64_t off = (uint64_t)(t - s.tile0) * tile_bytes(ul, THREADS) +
                                 ((uint64_t)threadIdx.x << ul);
            if (off >= s.bytes) continue;
            if (ul == 5) reduce_vector<T, ORDER, FAN_ALL, 32>(p, s, off, R, lpol, spol);
            else if (ul == 4) reduce_vector<T, ORDER, FAN_ALL, 16>(p, s, off, R, lpol, spol);
            else reduce_element<T, ORDER, FAN_ALL>(p, s, off, R);
            continue;
        }
        const uint64_t base = (uint64_t)(t - s.tile0) * tile_bytes(ul, THREADS * U);
        if (ul == 5) {
            reduce_tile<T, ORDER, FAN_ALL, 32, NR, THREADS>(p, s, base, R, lpol, spol);
        } else if (ul == 4) {
            reduce_tile<T, ORDER, FAN_ALL, 16, NR, THREADS>(p, s, base, R, lpol, spol);
        } else {
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint64_t off = base + ((uint64_t)(k * THREADS + threadIdx.x) << ul);
                if (off < s.bytes) reduce_element<T, ORDER, FAN_ALL>(p, s, off, R);
            }
        }
    }
}

// -------------------------------------------------------------------- copy

using atom::Unit;
using atom::load_unit;
using atom::store_unit;

template <int BYTES>
__device__ __forceinline__ void load_hinted(Unit<BYTES>& u, const char* p, uint64_t pol)
{
    if constexpr (BYTES >= 16) atom::load(u.v, p, pol);
    else load_unit<BYTES>(u, p);
}

template <int BYTES>
__device__ __forceinline__ void store_hinted(char* p, const Unit<BYTES>& u, uint64_t pol)
{
    if constexpr (BYTES >= 16) atom::store(p, u.v, pol);
    else store_unit<BYTES>(p, u);
}

// Atom::copy of one tile: UNROLL units per thread, each warp access
// contiguous; every unit loaded once and stored to one or all R outputs.
template <int BYTES, bool FAN_ALL, int THREADS, int UNROLL, int MAXSEG>
__device__ __forceinline__ void copy_tile(const ZsParams<MAXSEG>& p, const Segment& s,
                                          uint64_t base, uint64_t lpol, uint64_t spol)
{
    const uint64_t rem = s.bytes - base;
    const char* src = p.in[s.src] + s.src_off + base;
    Unit<BYTES> u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
        const uint64_t o = (uint64_t)(k * THREADS + threadIdx.x) * BYTES;
        if (o < rem) load_hinted<BYTES>(u[k], src + o, lpol);
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
        const uint64_t o = (uint64_t)(k * THREADS + threadIdx.x) * BYTES;
        if (o >= rem) continue;
        if (FAN_ALL) {
            for (int r = 0; r < (int)p.R; ++r) {
                char* dst = p.out[r] + s.dst_off + base + o;
                if (dst != src + o) store_hinted<BYTES>(dst, u[k], spol);  // in-place: skip
            }
        } else {
            store_hinted<BYTES>(p.out[s.dst] + s.dst_off + base + o, u[k], spol);
        }
    }
}

// THREADS x UNROLL units per tile: kThreads x kUnrollCopy for large messages,
// one warp with one unit per thread for small ones.  SHIFTED: as for the sums.
template <bool FAN_ALL, int MAXSEG, int THREADS, int UNROLL, bool SHIFTED>
__global__ void __launch_bounds__(THREADS, THREADS == kThreads ? 2 : 16)
zs_copy_kernel(const __grid_constant__ ZsParams<MAXSEG> p)
{
    pdl_enter();
    PURLIN_CHECK_BEGIN(p);
    const uint64_t lpol = atom::l2_policy(p.l2_load);
    const uint64_t spol = atom::l2_policy(p.l2_store);
    for (uint32_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const Segment& s = segment_of(p, t);
        const int ul = s.unit_log2;
        if constexpr (SHIFTED) {
            if (s.shift) {
                if (ul == 5) copy_shifted<32, FAN_ALL, THREADS, UNROLL>(p, s, t - s.tile0, lpol, spol);
                else copy_shifted<16, FAN_ALL, THREADS, UNROLL>(p, s, t - s.tile0, lpol, spol);
                continue;
            }
        }
        const uint64_t base = (uint64_t)(t - s.tile0) * tile_bytes(ul, THREADS * UNROLL);
        switch (ul) {
        case 5: copy_tile<32, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        case 4: copy_tile<16, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        case 3: copy_tile<8, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        case 2: copy_tile<4, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        case 1: copy_tile<2, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        default: copy_tile<1, FAN_ALL, THREADS, UNROLL>(p, s, base, lpol, spol); break;
        }
    }
}

// ------------------------------------------------------------ bulk copy
// Atom::copy through the Tensor Memory Accelerator: lane 0 of a one-warp CTA
// keeps a shared-memory ring of STAGES tiles busy -- cp.async.bulk
// global->shared loads that complete on an mbarrier, then one cp.async.bulk
// shared->global store per destination -- so a tile is read from HBM once and
// written R times without per-thread store instructions.  Half of the ring
// holds loads in flight ahead of the tile being stored, the other half tiles
// whose stores are still reading shared memory.  Tiles whose streams are not
// 16-byte aligned (unit < 16 B) are copied by the warp with ordinary accesses.

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for an mbarrier phase: at most ~2 s and 2^24 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    uint64_t start = 0;
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255) == 255) {
            const uint64_t t = global_ns();
            if (start == 0) start = t;
            else if (t - start > 2000000000ull) return false;
        }
    }
    return false;
}

__device__ __forceinline__ void bulk_load(void* smem, const char* gmem, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem)), "l"(gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_store(char* gmem, const void* smem, uint32_t bytes)
{
#if defined(PURLIN_CHECKED)
    if (!atom::access_ok(gmem, bytes, 16, false)) return;  // a bulk copy's run: 16-byte aligned
#endif
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(gmem), "r"(smem_u32(smem)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read_all_but()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int B, bool FAN_ALL, int MAXSEG>
__device__ __forceinline__ void warp_copy_tile(const ZsParams<MAXSEG>& p, const Segment& s,
                                               uint64_t base, uint64_t len)
{
    const char* src = p.in[s.src] + s.src_off + base;
    for (uint64_t o = (uint64_t)threadIdx.x * B; o < len; o += (uint64_t)kBulkThreads * B) {
        Unit<B> u;
        load_unit<B>(u, src + o);
        if (FAN_ALL) {
            for (int r = 0; r < (int)p.R; ++r) {
                char* dst = p.out[r] + s.dst_off + base + o;
                if (dst != src + o) store_unit<B>(dst, u);
            }
        } else {
            store_unit<B>(p.out[s.dst] + s.dst_off + base + o, u);
        }
    }
}

template <bool FAN_ALL, int MAXSEG, int STAGES>
__global__ void __launch_bounds__(kBulkThreads)
zs_copy_bulk_kernel(const __grid_constant__ ZsParams<MAXSEG> p)
{
    extern __shared__ __align__(128) char ring[];   // STAGES x kBulkStageBytes
    __shared__ __align__(8) uint64_t bar[STAGES];
    const uint32_t G = gridDim.x;
    pdl_enter();
    PURLIN_CHECK_BEGIN(p);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

        auto next_bulk = [&](uint32_t t) {
            while (t < p.ntiles && segment_of(p, t).unit_log2 < 4) t += G;
            return t;
        };
        auto tile_len = [&](uint32_t t, const Segment& s, uint64_t& base) {
            const uint64_t tb = tile_bytes(s.unit_log2, kTileUnitsBulk);
            base = (uint64_t)(t - s.tile0) * tb;
            return (uint32_t)min(tb, s.bytes - base);
        };
        auto issue_load = [&](uint32_t t, uint32_t n) {
            const Segment& s = segment_of(p, t);
            uint64_t base;
            const uint32_t len = tile_len(t, s, base);
            const int st = (int)(n % STAGES);
#if defined(PURLIN_CHECKED)
            if (!atom::access_ok(p.in[s.src] + s.src_off + base, len, 16, false)) {
                mbar_expect_tx(&bar[st], 0);  // skipped: the stage completes with no bytes
                return;
            }
#endif
            mbar_expect_tx(&bar[st], len);
            bulk_load(ring + (size_t)st * kBulkStageBytes, p.in[s.src] + s.src_off + base, len,
                      &bar[st]);
        };

        constexpr int AHEAD = STAGES / 2;
        uint32_t lt = next_bulk(blockIdx.x), stt = lt;
        uint32_t nl = 0, ns = 0;
        bool failed = false;
        while (nl < AHEAD && lt < p.ntiles) {
            issue_load(lt, nl++);
            lt = next_bulk(lt + G);
        }
        while (stt < p.ntiles) {
            const int st = (int)(ns % STAGES);
            if (!mbar_wait(&bar[st], (ns / STAGES) & 1u)) { failed = true; break; }
            const Segment& s = segment_of(p, stt);
            uint64_t base;
            const uint32_t len = tile_len(stt, s, base);
            const char* stage = ring + (size_t)st * kBulkStageBytes;
            if (FAN_ALL) {
                const char* src = p.in[s.src] + s.src_off + base;
                for (int r = 0; r < (int)p.R; ++r) {
                    char* dst = p.out[r] + s.dst_off + base;
                    if (dst != src) bulk_store(dst, stage, len);  // in-place block: skip
                }
            } else {
                bulk_store(p.out[s.dst] + s.dst_off + base, stage, len);
            }
            bulk_commit();
            ++ns;
            stt = next_bulk(stt + G);
            if (lt < p.ntiles) {
                // the slot being refilled was last read by the stores of tile
                // nl - STAGES: every store group but the newest STAGES - AHEAD
                // must have finished reading shared memory
                bulk_wait_read_all_but<STAGES - AHEAD>();
                issue_load(lt, nl++);
                lt = next_bulk(lt + G);
            }
        }
        if (failed) {
            atomicCAS(p.status, 0, (int)PURLIN_ERR_TIMEOUT);
            // every load already issued must land before shared memory is released
            for (uint32_t n = ns; n < nl; ++n) mbar_wait(&bar[n % STAGES], (n / STAGES) & 1u);
        }
        bulk_wait_all();
    }
    __syncwarp();

    for (uint32_t t = blockIdx.x; t < p.ntiles; t += G) {
        const Segment& s = segment_of(p, t);
        if (s.unit_log2 >= 4) continue;
        const uint64_t tb = tile_bytes(s.unit_log2, kTileUnitsBulk);
        const uint64_t base = (uint64_t)(t - s.tile0) * tb;
        const uint64_t len = min(tb, s.bytes - base);
        switch (s.unit_log2) {
        case 3: warp_copy_tile<8, FAN_ALL>(p, s, base, len); break;
        case 2: warp_copy_tile<4, FAN_ALL>(p, s, base, len); break;
        case 1: warp_copy_tile<2, FAN_ALL>(p, s, base, len); break;
        default: warp_copy_tile<1, FAN_ALL>(p, s, base, len); break;
        }
    }
}

}  // namespace
}  // namespace purlin
