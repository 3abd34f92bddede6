/*
 * purlin_layout.h -- host-only introspection of the layout module.
 *
 * The abstract of "Purlin: Separating Orchestration from the Datapath of
 * Collectives" derives coordination from "a naming of an input and output
 * layout"; Figure 4 gives the layouts.  purlin_plan_segments() exposes the plan
 * that the layout module derives from such a naming -- the exact list of
 * segments the Atom kernels will execute -- WITHOUT touching the GPU: the
 * buffer addresses are plain integers and are never dereferenced.  It exists so
 * that the plan (coverage of every output byte exactly once, alignment split,
 * tile numbering) can be tested on a machine with no GPU.
 */
#ifndef PURLIN_LAYOUT_H
#define PURLIN_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#include "purlin.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PURLIN_COLL_REDUCE_SCATTER = 0,
    PURLIN_COLL_ALL_GATHER = 1,
    PURLIN_COLL_ALL_REDUCE = 2,
    PURLIN_COLL_ALL_TO_ALL_V = 3
} purlin_collective_t;

/* One contiguous byte range of the plan. */
typedef struct {
    uint64_t src_off;  /* byte offset into the source buffer(s)                    */
    uint64_t dst_off;  /* byte offset into the destination buffer(s)               */
    uint64_t bytes;    /* length in bytes                                           */
    int32_t src_rank;  /* source rank, or -1: the same range of every input (sum)  */
    int32_t dst_rank;  /* destination rank, or -1: the same range of every output  */
    int32_t unit;      /* bytes per access: 32 or 16 (vector body), else element /
                          byte granularity for unaligned heads and tails            */
    uint32_t tile0;    /* first tile of the segment in the launch's tile space     */
    int32_t shift;     /* 0, or a shifted vector body: the destinations are aligned
                          to `unit`; the first source off that grid starts
                          `shift` bytes (0 < shift < unit) past a unit boundary.
                          The kernel reads aligned source blocks and realigns
                          them in registers (a sum realigns each rank on its own
                          offset, so its sources may sit on different grids).
                          A sum plan holding one has 16-byte bodies throughout  */
} purlin_segment_t;

/* Derive the plan of one collective.
 *   coll       which collective; arguments as in purlin.h:
 *                REDUCE_SCATTER: counts = recv_counts[R], displs_a = in_displs
 *                ALL_GATHER:     counts = counts[R],      displs_a = out_displs
 *                ALL_REDUCE:     count
 *                ALL_TO_ALL_V:   counts = send_counts[R*R], displs_a = send_displs,
 *                                displs_b = recv_displs
 *              Unused arguments may be NULL / 0.
 *   in_addr, out_addr  R integer addresses standing for the buffers.
 *   max_unit   widest access in bytes (16 or 32).
 *   segs       caller array of max_segs entries; *nsegs receives the count and
 *              *ntiles the number of tiles.  Tiles are those of the 256-thread
 *              zero-staging launch: 1024 units for copies; for sums in the fixed
 *              rank order 256 x U units, U = 4 for R <= 2, 2 for R = 3..4 and 1
 *              above (the pairwise order keeps U = 1, so its tiles differ); a
 *              shifted body's tiles hold 31/32 of those units (each warp's 32
 *              lanes write 31 units between the 32 source blocks they load); a call
 *              with fewer than the small-message threshold of them
 *              (purlin_set_small_tiles) runs one-warp tiles of 32 units over the
 *              same segments.
 * An AllGather whose outputs sit on different 16-byte alignments is planned by
 * destination (one piece per destination and source), as its launch is.  An
 * AllReduce whose outputs do is launched as a sum into output 0 followed by
 * copies to the others; the plan shown here is then the single fan-out plan.
 * Returns PURLIN_OK, PURLIN_ERR_INVALID_ARG (bad R, dtype, NULL array, element
 * misalignment for a sum, byte overflow) or PURLIN_ERR_UNSUPPORTED (more
 * segments than max_segs).  Never calls CUDA. */
PURLIN_API purlin_status_t purlin_plan_segments(purlin_collective_t coll, int R, const uint64_t in_addr[],
                                     const uint64_t out_addr[], const size_t counts[],
                                     const size_t displs_a[], const size_t displs_b[],
                                     size_t count, purlin_dtype_t dtype, int max_unit,
                                     purlin_segment_t* segs, int max_segs, int* nsegs,
                                     uint32_t* ntiles);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_LAYOUT_H */
