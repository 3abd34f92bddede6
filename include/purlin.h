/*
 * purlin.h -- C ABI of the Purlin copy/reduce datapath on one GB300 GPU.
 *
 * Source: the page "Purlin: Separating Orchestration from the Datapath of
 * Collectives".  Its abstract specifies a collective as "a naming of an input
 * and output layout and a copy or reduction operation"; Figure 4 gives the
 * layouts of ReduceScatter, AllGather and AllToAll on three ranks; Figure 6
 * composes AllReduce from ReduceScatter and AllGather; Table 2 marks the
 * variable-length "(V)" variants.  Here all R ranks are VIRTUAL: their buffers
 * all live in one GPU's memory, and every entry point moves data between those R
 * buffers with CUDA kernels on the caller's stream.
 *
 * General conventions (every entry point):
 *   - Buffers.  in[r] / out[r] are DEVICE pointers (from cudaMalloc or an
 *     allocator on top of it) for virtual rank r = 0..R-1.  The caller owns them
 *     and keeps them alive until the stream has passed the call.  A pointer may
 *     be NULL only when that rank's buffer has zero length in this call.
 *   - Host arrays (counts, displacements, pointer arrays) are read before the
 *     call returns and may be freed right after it.
 *   - Counts and displacements are in ELEMENTS of the call's dtype.  A NULL
 *     displacement array means the packed layout: partition k starts right
 *     after partitions 0..k-1, in rank order (Figure 4).
 *   - Asynchrony.  Calls enqueue kernels on `stream` and return without waiting.
 *     A handle may have one call in flight at a time (calls on one stream are
 *     naturally ordered); handles are not thread-safe.  The handle's device must
 *     be the current device of the calling thread.
 *   - Errors.  Argument errors return PURLIN_ERR_INVALID_ARG or
 *     PURLIN_ERR_UNSUPPORTED synchronously and enqueue nothing.  A failed launch
 *     returns PURLIN_ERR_CUDA.  Errors detected by a kernel (a bounded wait that
 *     timed out; in a checked build, an access outside the call's buffers) are
 *     recorded in the handle's device status word and reported by
 *     purlin_query_status() after the stream has been synchronized.
 *   - Aliasing.  Outputs must not overlap each other or any input, except for
 *     the in-place forms named at each entry point.
 *   - Reductions.  Every output element of a sum is a left fold over ranks
 *     0..R-1 in IEEE binary32 (round to nearest even), starting from rank 0's
 *     value, rounded once to the output dtype with round-to-nearest-even;
 *     subnormals are kept.  The result is bit-identical for every policy
 *     (variant, chunk size, pipeline depth, CTA count).  PURLIN_ORDER_TREE
 *     switches to a pairwise rank order instead.
 */
#ifndef PURLIN_H
#define PURLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PURLIN_MAX_RANKS 8

/* Symbols of this ABI are the only ones the shared library exports. */
#if defined(__GNUC__)
#define PURLIN_API __attribute__((visibility("default")))
#else
#define PURLIN_API
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* purlin_stream_t;

typedef enum {
    PURLIN_OK = 0,
    PURLIN_ERR_INVALID_ARG = 1,  /* bad pointer, size, overlap or handle        */
    PURLIN_ERR_UNSUPPORTED = 2,  /* valid request this library does not serve   */
    PURLIN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed        */
    PURLIN_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out          */
    PURLIN_ERR_OOM = 5,          /* device allocation failed (purlin_create)    */
    PURLIN_ERR_BOUNDS = 6        /* checked builds only: a kernel met an address
                                    outside the call's buffers and skipped it
                                    (purlin_debug.h)                           */
} purlin_status_t;

typedef enum {
    PURLIN_F32 = 0,   /* binary32: copy and sum                                */
    PURLIN_BF16 = 1,  /* bfloat16: copy and sum (binary32 accumulation)        */
    PURLIN_F16 = 2,   /* binary16: copy and sum (binary32 accumulation)        */
    PURLIN_U8 = 3     /* any 1-byte payload (e.g. fp8 codes): copy only        */
} purlin_dtype_t;

typedef enum { PURLIN_OP_COPY = 0, PURLIN_OP_SUM = 1 } purlin_op_t;

/* Which datapath runs a collective (a "codesign policy", Figure 1). */
typedef enum {
    PURLIN_VARIANT_AUTO = 0,    /* library's choice                               */
    PURLIN_VARIANT_ZS = 1,      /* zero staging: kernels read the sources directly
                                   (Figure 10, "Purlin-ZS omits staging")          */
    PURLIN_VARIANT_STAGED = 2,  /* SNAC: producers stage chunks into the handle's
                                   staging ring, notify through flags, consumers
                                   consume (abstract; Figure 6).  Sums stage the R
                                   input chunks and the consumer reduces them      */
    PURLIN_VARIANT_STAGED_Y = 3 /* SNAC as above, but for sums the producer reduces
                                   the R input chunks and stages the reduced chunk
                                   y, which the consumer copies to its destination
                                   (ReduceScatter) or to all R outputs (AllReduce);
                                   copies are staged as with PURLIN_VARIANT_STAGED */
} purlin_variant_t;

typedef enum {
    PURLIN_ORDER_FIXED = 0,  /* left fold over ranks 0..R-1 (default)           */
    PURLIN_ORDER_TREE = 1    /* pairwise: ((x0+x1)+(x2+x3))+((x4+x5)+(x6+x7)),
                                an odd last value carried up unchanged          */
} purlin_order_t;

/* Which mechanism moves the bytes of copy collectives (AllGather(V),
 * AllToAll(V)) on the zero-staging path.  The pages' Atom has one
 * specialization per GPU generation (Table 4) and note that one AllGather
 * baseline "uses the copy engine and launches no kernel" (Figure 10). */
typedef enum {
    PURLIN_ATOM_AUTO = 0,         /* library's choice (measured best: VECTOR)        */
    PURLIN_ATOM_VECTOR = 1,       /* every thread moves 16/32-byte vectors           */
    PURLIN_ATOM_BULK = 2,         /* one thread per CTA drives TMA bulk copies
                                     (cp.async.bulk) through a shared-memory ring   */
    PURLIN_ATOM_COPY_ENGINE = 3   /* no kernel: one cudaMemcpyAsync per block and
                                     destination, on the copy engines               */
} purlin_atom_t;

/* How an AllGather's copies are organized (push vs pull, Figures 7 and 11).
 * PUSH: work is split by source tile; a tile is read once and written to all R
 * destinations.  PULL: work is split by destination; each destination pulls
 * every source's block (R reads of each source, from L2 after the first). */
typedef enum {
    PURLIN_DIRECTION_AUTO = 0,  /* library's choice: PUSH (measured best), PULL
                                   when the outputs sit on different 16-byte
                                   alignments (then one push body cannot be
                                   aligned to all of them)                     */
    PURLIN_DIRECTION_PUSH = 1,
    PURLIN_DIRECTION_PULL = 2
} purlin_direction_t;

typedef struct purlin_handle* purlin_handle_t;
typedef struct purlin_plan* purlin_plan_t;

/* What the last collective on a handle launched (for SM accounting, Figure 10:
 * concurrent SM use is bounded by min(CTAs launched, SMs)). */
typedef struct {
    int variant;          /* PURLIN_VARIANT_ZS or PURLIN_VARIANT_STAGED       */
    int kernels;          /* kernel launches made by the call                 */
    int grid;             /* CTAs of the (largest) launch                     */
    int block;            /* threads per CTA                                  */
    int sms;              /* SMs on the device                                */
    int depth;            /* SNAC ring slots per channel (0 for ZS)           */
    size_t chunk_bytes;   /* SNAC chunk, or the ZS tile, in bytes             */
    size_t bytes_moved;   /* algorithmic bytes: read + written by the call    */
} purlin_launch_info_t;

/* ------------------------------------------------------------------------- */
/* Handle                                                                     */
/* ------------------------------------------------------------------------- */

/* Create a handle for R virtual ranks (1..PURLIN_MAX_RANKS) on CUDA device
 * `device`.  The handle owns the SNAC staging ring (staging_bytes; 0 picks
 * 64 MiB, half the L2 cache: room for a channel on every resident CTA pair at
 * the default chunks of 8 ranks), its ready/free flags and a device
 * status word, all allocated here with cudaMalloc (PURLIN_ERR_OOM on failure).
 * On success *h receives the handle; on failure *h is set to NULL.
 * Environment, read here, for measurements and sweeps only (the defaults are the
 * measured best; a value out of range is ignored): PURLIN_CHUNK, PURLIN_DEPTH,
 * PURLIN_CTAS and PURLIN_VARIANT set the initial policy as purlin_set_policy
 * would; PURLIN_SMALL_TILES as purlin_set_small_tiles; PURLIN_PDL (0 turns
 * programmatic dependent launch off); PURLIN_L2_LOAD / PURLIN_L2_STORE and
 * PURLIN_L2_<RS|AG|AR|A2A>_<LOAD|STORE> (0 normal, 1 evict-first, 2 evict-last)
 * set the L2 priority of the zero-staging kernels' streams; PURLIN_MAX_UNIT
 * (2..32 bytes) caps their vector unit. */
PURLIN_API purlin_status_t purlin_create(purlin_handle_t* h, int R, size_t staging_bytes, int device);

/* Synchronize the device, free everything the handle owns, free the handle.
 * NULL is accepted and ignored. */
PURLIN_API purlin_status_t purlin_destroy(purlin_handle_t h);

/* ------------------------------------------------------------------------- */
/* Collectives (Figure 4 layouts; Table 2 "(V)" variants)                     */
/* ------------------------------------------------------------------------- */

/* ReduceScatter(V), Figure 4 (top): partition k of every input is summed into
 * y_k at rank k.
 *   in[r]        R device pointers; partition k of rank r is the
 *                recv_counts[k] elements at in[r] + in_displs[k] (packed when
 *                in_displs is NULL).  Every rank uses the same partitioning.
 *   out[k]       R device pointers; out[k] receives recv_counts[k] elements.
 *   recv_counts  R counts (host); zero allowed.
 *   dtype        PURLIN_F32, PURLIN_BF16 or PURLIN_F16; every pointer aligned to
 *                the element size.
 *   op           PURLIN_OP_SUM (PURLIN_OP_COPY: PURLIN_ERR_UNSUPPORTED).
 *   In-place: out[k] == in[k] + in_displs[k] (rank k's own partition) is allowed.
 */
PURLIN_API purlin_status_t purlin_reduce_scatter(purlin_handle_t h, const void* const in[],
                                      void* const out[], const size_t recv_counts[],
                                      const size_t in_displs[], purlin_dtype_t dtype,
                                      purlin_op_t op, purlin_stream_t stream);

/* AllGather(V), Figure 4 (top): every rank receives every rank's block, placed
 * in rank order.
 *   in[k]        R device pointers; in[k] holds counts[k] elements.
 *   out[j]       R device pointers; out[j] + out_displs[k] receives in[k]
 *                (packed when out_displs is NULL).  Blocks must not overlap.
 *   counts       R counts (host); zero allowed.
 *   dtype        any; only its size matters (a copy moves bytes).
 *   In-place: in[k] == out[k] + out_displs[k] is allowed.
 */
PURLIN_API purlin_status_t purlin_all_gather(purlin_handle_t h, const void* const in[],
                                  void* const out[], const size_t counts[],
                                  const size_t out_displs[], purlin_dtype_t dtype,
                                  purlin_stream_t stream);

/* AllReduce, Figure 6 (AllGather composed with ReduceScatter): every out[j]
 * receives the sum over ranks of the `count` elements of in[0..R-1].
 *   dtype        PURLIN_F32, PURLIN_BF16 or PURLIN_F16.
 *   op           PURLIN_OP_SUM.
 *   In-place: out[r] == in[r] for every r is allowed.
 * Zero staging runs one kernel that writes each sum to all R outputs; when the
 * outputs sit on different 16-byte alignments it runs two, in stream order: the
 * sum into out[0], then copies of out[0] to the other outputs.
 */
PURLIN_API purlin_status_t purlin_all_reduce(purlin_handle_t h, const void* const in[],
                                  void* const out[], size_t count, purlin_dtype_t dtype,
                                  purlin_op_t op, purlin_stream_t stream);

/* AllToAll, Figure 4 (bottom): rank j receives partition j of every source s,
 * in source order; every partition holds count_per_pair elements.  This is
 * purlin_all_to_all_v with equal counts and packed layouts.  No in-place form. */
PURLIN_API purlin_status_t purlin_all_to_all(purlin_handle_t h, const void* const in[],
                                  void* const out[], size_t count_per_pair,
                                  purlin_dtype_t dtype, purlin_stream_t stream);

/* AllToAllV, Figure 4 (bottom) with Table 2's variable lengths:
 *   send_counts  R*R counts (host), [s*R + j] = elements from source s to rank j.
 *   send_displs  R*R (host), [s*R + j] = where that block starts in in[s];
 *                NULL = packed per source in destination order.
 *   recv_displs  R*R (host), [j*R + s] = where it lands in out[j];
 *                NULL = packed per destination in source order.
 *   dtype        any; only its size matters.  Received blocks must not overlap.
 *   No in-place form. */
PURLIN_API purlin_status_t purlin_all_to_all_v(purlin_handle_t h, const void* const in[],
                                    void* const out[], const size_t send_counts[],
                                    const size_t send_displs[], const size_t recv_displs[],
                                    purlin_dtype_t dtype, purlin_stream_t stream);

/* AllReduce that allocates nothing.  The paper has no counterpart to this call.
 *
 * Some callers cannot call cudaMalloc: a host framework that has reserved the
 * GPU's memory for its own pool (a direct cudaMalloc would fail or escape its
 * accounting), a plugin that may not own device memory, or a latency-critical
 * path that cannot take the synchronization cudaMalloc/cudaFree may cause.  The
 * handle-based calls above allocate their scratch in purlin_create(); this one
 * needs no handle.  It runs the staged (SNAC) AllReduce kernel that stages the
 * reduced chunk (PURLIN_VARIANT_STAGED_Y) -- same result, bit for bit, as
 * purlin_all_reduce -- with its staging ring, flags and status word in one
 * static device array of PURLIN_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU
 * which loads this library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   in, out      R device pointers each; out[r] == in[r] (in-place) is allowed,
 *                any other overlap is PURLIN_ERR_INVALID_ARG.
 *   R            1..PURLIN_MAX_RANKS;  count: elements per rank.
 *   dtype        PURLIN_F32, PURLIN_BF16 or PURLIN_F16.
 *   chunk_bytes  staged bytes per rank per pipeline step, a multiple of 256
 *                (0 = 8 KiB); depth: ring slots, 0..8 (0 = 2).  A channel's
 *                ring that cannot fit in the static array -- depth * chunk_bytes
 *                above PURLIN_NOALLOC_SCRATCH_BYTES - 64 KiB -- is rejected with
 *                PURLIN_ERR_INVALID_ARG before anything is enqueued; the array
 *                holds as many channels as fit (508 at the defaults).
 *   device_status  optional DEVICE int: set to 0 on the stream, then to
 *                PURLIN_ERR_TIMEOUT if a bounded wait of the kernel ran out
 *                (NULL: the library's own word inside the static array is used
 *                and not reported).
 *   stream       runs on the current device, on this stream.
 * The first call on a device looks up the static array's device address (with
 * that device current); make that first call before any stream capture.  If
 * the lookup fails the call returns PURLIN_ERR_CUDA having enqueued nothing,
 * and the next call on that device tries the lookup again.  Every
 * call on a device shares the one array: calls whose kernels overlap on the GPU
 * (e.g. on two streams at once) race and produce wrong results; serialize them.
 * Flags hold per-call epoch tags and the status word is cleared at each call, so
 * what the last call left behind needs no other clearing. */
#define PURLIN_NOALLOC_SCRATCH_BYTES (8u << 20)
PURLIN_API purlin_status_t purlin_all_reduce_noalloc(const void* const in[], void* const out[],
                                                     int R, size_t count, purlin_dtype_t dtype,
                                                     size_t chunk_bytes, int depth,
                                                     int* device_status, purlin_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Plans: check and lay out a collective once, launch it many times           */
/* ------------------------------------------------------------------------- */

/* The layout module turns a collective's naming into a plan (Figure 1:
 * collectives are "a naming of an input and output layout"); these calls keep
 * that plan so that a call repeated on the same buffers costs one launch.
 *
 * purlin_plan_begin(h): the NEXT collective call on h (any entry point above
 * that takes h) is checked and planned exactly as usual, with h's policy at that
 * moment, but enqueues nothing.  A second collective call before
 * purlin_plan_end returns PURLIN_ERR_INVALID_ARG.  Errors of the recorded call
 * are returned by that call, as usual.
 * purlin_plan_end(h, &plan): *plan receives the recorded call (NULL and
 * PURLIN_ERR_INVALID_ARG if none was recorded).  Recording stops either way.
 * purlin_plan_launch(plan, stream): enqueue the planned call on `stream`; same
 * kernels, same parameters, same result bit for bit as the direct call.  The
 * buffers, counts and displacements are those of the recorded call: the caller
 * keeps the buffers alive and the plan sees whatever they hold at launch time.
 * The plan uses h's staging ring, flags and status word (staged calls), so h
 * must outlive it, and launches of plans and calls of one handle must not
 * overlap on the GPU (as for any call on h).  Safe to capture in a CUDA graph.
 * purlin_plan_destroy(plan): free the plan (host memory only); NULL is
 * ignored. */
PURLIN_API purlin_status_t purlin_plan_begin(purlin_handle_t h);
PURLIN_API purlin_status_t purlin_plan_end(purlin_handle_t h, purlin_plan_t* plan);
PURLIN_API purlin_status_t purlin_plan_launch(purlin_plan_t plan, purlin_stream_t stream);
PURLIN_API purlin_status_t purlin_plan_destroy(purlin_plan_t plan);

/* ------------------------------------------------------------------------- */
/* Policy, status, introspection                                              */
/* ------------------------------------------------------------------------- */

/* Codesign policy (Figure 1; chunk sizing after Table 3's bandwidth-delay
 * products; depth after Figure 11).  0 for any argument keeps the automatic
 * choice.
 *   chunk_bytes  SNAC bytes per rank per pipeline step, a multiple of 16 (the
 *                staged kernels round it up to a multiple of 256).  A staged call
 *                whose ring cannot hold one channel -- depth x chunk x (R + 1 for
 *                an AllReduce staging its inputs, R for a ReduceScatter staging
 *                its inputs, 1 for copies and for sums staging the reduced
 *                chunk) above the handle's staging bytes -- returns
 *                PURLIN_ERR_UNSUPPORTED.
 *   depth        SNAC ring slots per channel, 1..8.
 *   ctas         0..65535: CTAs per zero-staging launch (automatic: 16 per
 *                resident CTA slot of the device, 4 for the TMA bulk Atom, at
 *                most one per tile), or SNAC channels (CTAs per role; a role
 *                CTA has 64 threads, up to 8 per SM: automatic is every channel
 *                the residency, the ring and the flags allow).
 *   variant      a purlin_variant_t.
 * Out-of-range values: PURLIN_ERR_INVALID_ARG. */
PURLIN_API purlin_status_t purlin_set_policy(purlin_handle_t h, size_t chunk_bytes, int depth,
                                  int ctas, int variant);

/* Mechanism of copy collectives on the zero-staging path: a purlin_atom_t.
 * Sums always run on the vector Atom; the staged path ignores this setting. */
PURLIN_API purlin_status_t purlin_set_atom(purlin_handle_t h, int atom);

/* Push or pull organization of AllGather(V) copies on the zero-staging path
 * (a purlin_direction_t).  Other collectives ignore it. */
PURLIN_API purlin_status_t purlin_set_direction(purlin_handle_t h, int direction);

/* Launch shape of zero-staging kernels by message size.  A call whose
 * large-message plan has fewer than `tiles` tiles runs one-warp CTAs with one
 * access unit per thread instead of 256-thread CTAs, so that a message of a few
 * KiB is spread over many SMs rather than queued in the load/store path of one
 * (a tile here: 256 threads x one 16/32-byte unit for sums, counted so also
 * where sums of 2 to 4 ranks run larger tiles; x four units for copies; the TMA
 * bulk Atom always runs its own shape).  tiles = 0: never;
 * tiles = -1: the library default, per collective (measured on GB300: 256 for
 * AllReduce, 64 for the others).  Other negative values:
 * PURLIN_ERR_INVALID_ARG. */
PURLIN_API purlin_status_t purlin_set_small_tiles(purlin_handle_t h, int tiles);

/* Rank order of sums: PURLIN_ORDER_FIXED (default) or PURLIN_ORDER_TREE. */
PURLIN_API purlin_status_t purlin_set_reduce_order(purlin_handle_t h, int order);

/* Limit of every bounded device-side wait of the SNAC kernels, in nanoseconds
 * (default 1e9).  When a wait runs out the kernel records PURLIN_ERR_TIMEOUT in
 * the status word, every CTA leaves its loop, and the kernel returns. */
PURLIN_API purlin_status_t purlin_set_timeout(purlin_handle_t h, uint64_t timeout_ns);

/* Read and clear the device status word.  Call after synchronizing the stream
 * of the last call; returns PURLIN_OK or the first error a kernel recorded. */
PURLIN_API purlin_status_t purlin_query_status(purlin_handle_t h);

/* What the last collective on `h` launched. */
PURLIN_API purlin_status_t purlin_last_launch(purlin_handle_t h, purlin_launch_info_t* info);

/* Static English text for a status code. */
PURLIN_API const char* purlin_status_string(purlin_status_t s);

/* Version of this ABI, (major << 16) | minor. */
PURLIN_API int purlin_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_H */
