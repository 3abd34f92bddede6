// internal.h -- declarations shared by the C-ABI layer and the kernel
// translation units of the CUDA library.
#pragma once

#include <cuda_runtime.h>

#include "check.h"
#include "plan.h"

namespace purlin {

// Element type codes (the values of purlin_dtype_t).
enum : int { kF32 = 0, kBF16 = 1, kF16 = 2, kU8 = 3 };

// ---- one kernel launch, fully planned --------------------------------------
// The C-ABI layer builds a call's kernel parameters directly in `params`, the
// kernel translation units fill in the function and its launch shape, and the
// launch is then either made at once or kept in a plan and made many times.

constexpr size_t kMaxLaunchParams = 8192;

struct KernelLaunch {
    const void* func = nullptr;
    unsigned grid = 0;
    unsigned block = 0;
    size_t smem = 0;
    bool pdl = false;          // programmatic stream serialization
    bool cooperative = false;  // every CTA resident at once
    size_t params_bytes = 0;
    alignas(16) unsigned char params[kMaxLaunchParams];
};

// Launch k on `stream` (its parameter block passed by value).
cudaError_t launch_kernel(const KernelLaunch& k, cudaStream_t stream);

// Resident CTAs per SM of `kernel` at `threads` threads and no dynamic shared
// memory, on the current device (occupancy API, cached without allocating; 1
// if the query fails).
int resident_ctas_of(const void* kernel, int threads);

// ---- device status area and checked builds ----------------------------------
// A handle's (or the allocation-free call's) status area: the status word, then
// the first address a checked kernel met outside the call's buffers.
constexpr size_t kStatusBytes = 16;

inline unsigned long long* violation_word(int* status)
{
    return reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(status) + 8);
}

// The address ranges of a call's buffers: input r is [in[r], in[r] + in_ext[r]),
// output r [out[r], out[r] + out_ext[r]) (empty extents left out).
CheckRanges call_ranges(int R, const uint64_t* in, const uint64_t* out, const uint64_t* in_ext,
                        const uint64_t* out_ext, unsigned long long* bad);

// Appends [lo, lo + bytes) to c (if there is room).
void add_range(CheckRanges& c, uint64_t lo, uint64_t bytes);

// ---- zero-staging Atom kernels (zs_kernels.cu) -----------------------------

// Each *_select call fills k's function, block, dynamic shared memory and
// parameter size for a parameter block already built in k.params; the caller
// sets the grid and pdl.

// Sum over ranks.  fan_all: write each result to every output (AllReduce),
// else to the segment's destination (ReduceScatter).  small: one-warp CTAs, plan
// built with kTileUnitsSmall; else kThreads-thread CTAs, kTileUnitsReduce.
// Units per thread of the kThreads-thread sum kernel for R ranks and a rank
// order (R x units <= kMaxRanks vectors in flight per thread); the plan's tiles
// are kThreads x reduce_unroll(R, order) units.  shift_mode: 0 the plan holds
// no shifted segment (Segment::shift); 1 shifted segments whose sources share
// one offset; 2 one whose ranks' sources sit on different offsets (kernels of
// the fixed rank order only serve 1 and 2).
int reduce_unroll(int R, int order);
void zs_reduce_select(KernelLaunch& k, int dtype, int order, bool fan_all, bool small, int R,
                      int shift_mode);
int zs_reduce_resident_ctas(int dtype, int order, bool fan_all, bool small, int R, int shift_mode);

// Copy.  fan_all: every segment goes to every output (AllGather), else to the
// segment's destination (AllToAll(V)).  large: ZsParams<kSegsLarge> (else
// kSegsSmall).  small: one-warp CTAs, plan built with kTileUnitsSmall; else
// kThreads-thread CTAs, kTileUnitsCopy.  shifted: as for the sums.
void zs_copy_select(KernelLaunch& k, bool large, bool fan_all, bool small, bool shifted);
int zs_copy_resident_ctas(bool large, bool fan_all, bool small, bool shifted);

// Copy through TMA bulk transfers (plan built with kTileUnitsBulk tiles).
// Returns the CUDA error of the one-time shared-memory opt-in, if any.
cudaError_t zs_copy_bulk_select(KernelLaunch& k, bool large, bool fan_all);
int zs_copy_bulk_resident_ctas(bool large, bool fan_all);

}  // namespace purlin
