// internal.h -- declarations shared by the C-ABI layer and the kernel
// translation units of the CUDA library.
#pragma once

#include <cuda_runtime.h>

#include "plan.h"

namespace purlin {

// Element type codes (the values of purlin_dtype_t).
enum : int { kF32 = 0, kBF16 = 1, kF16 = 2, kU8 = 3 };

// ---- zero-staging Atom kernels (zs_kernels.cu) -----------------------------

// Sum over ranks.  fan_all: write each result to every output (AllReduce),
// else to the segment's destination (ReduceScatter).  small: one-warp CTAs, plan
// built with kTileUnitsSmall; else kThreads-thread CTAs, kTileUnitsReduce.
cudaError_t zs_reduce_launch(const ZsParams<kSegsSmall>& p, int dtype, int order, bool fan_all,
                             bool small, int grid, cudaStream_t stream);
int zs_reduce_resident_ctas(int dtype, int order, bool fan_all, bool small);

// Copy.  fan_all: every segment goes to every output (AllGather), else to the
// segment's destination (AllToAll(V)).  small: one-warp CTAs, plan built with
// kTileUnitsSmall; else kThreads-thread CTAs, kTileUnitsCopy.
cudaError_t zs_copy_launch(const ZsParams<kSegsSmall>& p, bool fan_all, bool small, int grid,
                           cudaStream_t stream);
cudaError_t zs_copy_launch(const ZsParams<kSegsLarge>& p, bool fan_all, bool small, int grid,
                           cudaStream_t stream);
int zs_copy_resident_ctas(bool large, bool fan_all, bool small);

// Copy through TMA bulk transfers (plan built with kTileUnitsBulk tiles).
cudaError_t zs_copy_bulk_launch(const ZsParams<kSegsSmall>& p, bool fan_all, int grid,
                                cudaStream_t stream);
cudaError_t zs_copy_bulk_launch(const ZsParams<kSegsLarge>& p, bool fan_all, int grid,
                                cudaStream_t stream);
int zs_copy_bulk_resident_ctas(bool large, bool fan_all);

}  // namespace purlin
