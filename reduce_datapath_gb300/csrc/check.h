// check.h -- the address ranges of a call, for the library's checked build.
//
// Checked builds (compiled with PURLIN_CHECKED): the address ranges a launch
// may touch -- its inputs, its outputs and, for the staged kernels, the
// staging ring.  Every global access of an Atom is tested against them first;
// one outside all of them is skipped, and the first such address is recorded
// in *bad (and PURLIN_ERR_BOUNDS in the status word).  The product build
// carries none of this in its kernels.
#pragma once

#include <cstdint>

namespace purlin {

// Inputs and outputs of up to 8 ranks, and a staging ring.
constexpr int kMaxCheckRanges = 17;

struct CheckRanges {
    uint64_t lo[kMaxCheckRanges];
    uint64_t hi[kMaxCheckRanges];   // exclusive
    uint32_t n;
    uint32_t pad;
    unsigned long long* bad;
};

}  // namespace purlin
