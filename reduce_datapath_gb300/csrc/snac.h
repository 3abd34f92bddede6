// snac.h -- host interface of the SNAC (Stage, Notify, And Consume) kernels.
//
// Page "Purlin: Separating Orchestration from the Datapath of Collectives":
// the abstract introduces SNAC as the shared orchestration protocol derived
// from the collective's layouts; Figure 6 shows the composed AllReduce in which
// every rank stages chunks incrementally while partition k is reduced and
// already-reduced chunks are gathered.  On one GPU the protocol runs inside one
// cooperative launch:
//   producer CTAs  stage a chunk of every source into a slot of the staging
//                  ring, then NOTIFY with a release store of the step's tag;
//   consumer CTAs  acquire the tag (bounded wait), CONSUME the slot -- sum the
//                  R staged pieces, or copy the staged piece -- into the
//                  destination(s) or, for AllReduce, into the slot's y part,
//                  then release the slot back to the producer;
//   gatherer CTAs  (AllReduce) acquire the y tag and copy the reduced chunk to
//                  all R outputs (the AllGather half of Figure 6).
// Each CHANNEL is one producer, one consumer (and one gatherer) with its own
// ring of `depth` slots; steps (chunks) are handed to channels from a device
// counter as their producers ask for them.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"
#include "plan.h"
#include "purlin.h"

namespace purlin {

struct SnacRequest {
    Coll coll;
    int R;
    int dtype;
    int order;
    size_t esz;
    const Piece* pieces;
    int npieces;
    uint64_t in[kMaxRanks];
    uint64_t out[kMaxRanks];
    bool stage_y;  // sums: the producer reduces and stages the reduced chunk
#if defined(PURLIN_CHECKED)
    const CheckRanges* check;  // the call's buffers
#endif
};

struct SnacConfig {
    char* staging;          // device ring memory (owned by the caller)
    size_t staging_bytes;
    uint64_t* flags;        // device flag words, zeroed once at creation; the last
                            // two hold the device epoch and a completion counter
    size_t flag_words;
    int* status;            // device status word (0 = ok)
    size_t chunk_bytes;     // 0 = automatic
    int depth;              // 0 = automatic
    int channels;           // 0 = automatic
    int sms;
    uint64_t timeout_ns;
    int inject_skip_notify; // testing: channel 0's producer never notifies step 0
};

struct SnacLaunch {
    int kernels;
    int grid;
    int block;
    int depth;
    int channels;
    size_t chunk_bytes;
};

// Plan one staged call: the cooperative kernel, its launch shape and its
// parameter block in k (k.grid = 0: nothing to launch).  Launch with
// launch_kernel (internal.h), once or many times.
purlin_status_t snac_plan(const SnacRequest& rq, const SnacConfig& cfg, KernelLaunch& k,
                          SnacLaunch* launch);

// Plan and launch at once, with the parameter block on the caller's stack (no
// memory is allocated).
purlin_status_t snac_run_on_stack(const SnacRequest& rq, const SnacConfig& cfg,
                                  cudaStream_t stream, SnacLaunch* launch);

// Channels, chunk and depth that snac_plan would choose.
purlin_status_t snac_geometry(int R, Coll coll, bool stage_y, const SnacConfig& cfg,
                              int resident_per_sm, uint64_t total_bytes, size_t* chunk,
                              int* depth, int* channels);

}  // namespace purlin
