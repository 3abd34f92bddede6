// plan.h -- the per-call plan that the layout module derives from a collective's
// naming and that the Atom kernels execute.  Shared by host and device code of
// the CUDA library (never by the oracle).
//
// A collective (page "Purlin: Separating Orchestration from the Datapath of
// Collectives", abstract and Figure 4) is a naming of input and output
// partitions plus an operation.  The layout module turns it into a list of
// SEGMENTS: contiguous byte ranges that go from one source buffer (copy) or from
// the same offset of every source buffer (sum) to one destination buffer or to
// the same offset of every destination buffer.  Each segment is executed with
// one access width ("unit"): a 16- or 32-byte vector for aligned bodies, or the
// element / byte for unaligned heads and tails.  The launch's work is a flat
// space of TILES (one tile = tile_units units: the threads of a CTA x units per
// thread); a segment owns the tiles [tile0, tile0 + its tile count).
#pragma once

#include <cstddef>
#include <cstdint>

#if defined(PURLIN_CHECKED)
#include "check.h"
#endif

#if defined(__CUDACC__)
#define PURLIN_HD __host__ __device__
#else
#define PURLIN_HD
#endif

namespace purlin {

constexpr int kMaxRanks = 8;
constexpr int kThreads = 256;          // threads per CTA of every Atom kernel
constexpr uint8_t kEveryRank = 0xff;   // src: sum over all ranks; dst: all outputs
constexpr int kSegsSmall = 24;         // RS / AG / AR: <= 3 segments per rank
constexpr int kSegsLarge = 3 * kMaxRanks * kMaxRanks;  // A2AV: <= 3 per pair
constexpr int kUnrollReduce = 1;       // units per thread per tile, sums
constexpr int kUnrollCopy = 4;         // units per thread per tile, copies
// Units per tile of the large-message launches (kThreads threads per CTA).
constexpr int kTileUnitsReduce = kThreads * kUnrollReduce;
constexpr int kTileUnitsCopy = kThreads * kUnrollCopy;
// Small messages run one-warp CTAs with one unit per thread, so that a few KiB
// spread over many SMs instead of queueing in one.
constexpr int kSmallThreads = 32;
constexpr int kTileUnitsSmall = kSmallThreads;

struct Segment {
    uint64_t src_off;   // byte offset in the source buffer(s)
    uint64_t dst_off;   // byte offset in the destination buffer(s)
    uint64_t bytes;     // length; a multiple of the unit
    uint32_t tile0;     // first tile of this segment
    uint8_t src;        // source rank, or kEveryRank (sum over ranks)
    uint8_t dst;        // destination rank, or kEveryRank (every output)
    uint8_t unit_log2;  // access width = 1 << unit_log2 bytes (0..5)
    uint8_t shift;      // 0, or a shifted body: destinations aligned to the unit,
                        // every source `shift` bytes past a unit boundary; with
                        // kShiftPerRank set (sums), the sources sit on different
                        // offsets (the low bits: the first non-zero one), which
                        // the kernel reads from their addresses
};

constexpr uint8_t kShiftPerRank = 0x80;
static_assert(sizeof(Segment) == 32, "Segment is passed by value to kernels");

#if defined(PURLIN_CHECKED)
static_assert(kMaxCheckRanges >= 2 * kMaxRanks + 1, "check ranges");
#endif

// Kernel parameter block of the zero-staging Atom kernels (passed as a
// __grid_constant__ argument: no host-to-device copy per call).
// L2 eviction priority of a stream (PTX createpolicy).
enum : uint32_t { kL2Normal = 0, kL2EvictFirst = 1, kL2EvictLast = 2 };

template <int MAXSEG>
struct ZsParams {
    const char* in[kMaxRanks];
    char* out[kMaxRanks];
    uint32_t l2_load;   // eviction priority of source loads (kL2*)
    uint32_t l2_store;  // ... and of destination stores
    uint32_t pdl;       // launched with programmatic stream serialization
    int* status;        // device status word (bounded waits of the bulk kernel, plan checks)
    uint32_t R;
    uint32_t nseg;
    uint32_t ntiles;
    uint32_t tile_units;  // units per tile
#if defined(PURLIN_CHECKED)
    CheckRanges check;
#endif
    Segment seg[MAXSEG];
};

// Tile length in bytes of a segment with this unit.
PURLIN_HD inline uint64_t tile_bytes(int unit_log2, int tile_units)
{
    return (uint64_t)tile_units << unit_log2;
}

// Units per tile of a shifted segment: each warp's 32 lanes load 32 aligned
// source blocks and write the 31 destination units that lie between them (a
// destination unit takes the tail of one source block and the head of the next).
PURLIN_HD constexpr int shifted_tile_units(int tile_units)
{
    return tile_units / 32 * 31;
}

constexpr int kUnrollBulk = 2;          // bulk-copy tiles: 256 x unit x 2 bytes (<= 16 KiB)
constexpr int kTileUnitsBulk = kThreads * kUnrollBulk;
constexpr int kBulkThreads = 32;        // one warp per bulk-copy CTA
constexpr uint32_t kBulkStageBytes = 16 * 1024;

enum class Coll : int { ReduceScatter = 0, AllGather = 1, AllReduce = 2, AllToAllV = 3 };

// A piece of a collective before alignment splitting.
struct Piece {
    uint64_t src_off;
    uint64_t dst_off;
    uint64_t bytes;
    uint8_t src;
    uint8_t dst;
};

// ---- layout module (layout.cpp; host only) ---------------------------------

// Logical pieces of a collective from its counts and displacements (elements).
//   ReduceScatter: counts = recv_counts[R], da = in_displs   (NULL = packed)
//   AllGather:     counts = counts[R],      da = out_displs  (NULL = packed)
//   AllReduce:     count
//   AllToAllV:     counts = send_counts[R*R], da = send_displs, db = recv_displs
// Returns the number of pieces (zero-length ones dropped), or -1 on overflow
// of 64-bit byte arithmetic.
int layout_pieces(Coll coll, int R, const size_t* counts, const size_t* da,
                  const size_t* db, size_t count, size_t elem_bytes, Piece* out, int max_out);

// Byte extent [0, extent) touched in every input and output buffer.
void layout_extents(Coll coll, int R, const size_t* counts, const size_t* da,
                    const size_t* db, size_t count, size_t elem_bytes,
                    uint64_t in_extent[kMaxRanks], uint64_t out_extent[kMaxRanks]);

// Split pieces into head / body / tail segments by the alignment of the actual
// addresses, then number the tiles (tile_units x unit bytes each;
// shifted_tile_units for a shifted body).  `reduce` selects element-wise heads
// and tails (sums) or byte-wise ones (copies).  max_unit_log2 caps the vector
// width (4 = 16 B, 5 = 32 B).  When the sources and the destinations of a piece
// cannot share one vector alignment but each side agrees within itself,
// `allow_shift` gives the body vector units aligned to the destinations and a
// source shift (Segment::shift) instead of element or byte units.  Returns the
// segment count or -1 if max_segs is too small; *ntiles receives the tile count.
int layout_segments(const Piece* pieces, int npieces, int R, const uint64_t* in_addr,
                    const uint64_t* out_addr, size_t elem_bytes, bool reduce, int tile_units,
                    int max_unit_log2, bool allow_shift, Segment* segs, int max_segs,
                    uint32_t* ntiles);

}  // namespace purlin
