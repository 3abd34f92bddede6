/*
 * purlin_debug.h -- fault injection for testing the bounded waits, and the
 * checked build's access records.
 *
 * The SNAC protocol ("Purlin: Separating Orchestration from the Datapath of
 * Collectives", abstract; Figure 6) makes consumers wait on flags that producers
 * publish.  Every such wait in this library is bounded (purlin_set_timeout).  This
 * hook lets a test make one wait run out on purpose WITHOUT faulting or hanging
 * the GPU: the flag simply never gets its value, the waiting CTA records
 * PURLIN_ERR_TIMEOUT in the handle's status word after the timeout, every other
 * CTA leaves at its next wait, and the kernel returns normally.
 */
#ifndef PURLIN_DEBUG_H
#define PURLIN_DEBUG_H

#include <stdint.h>

#include "purlin.h"

#ifdef __cplusplus
extern "C" {
#endif

/* what = 1: in the NEXT staged (PURLIN_VARIANT_STAGED) call on h, the producer
 * of channel 0 stages its first chunk but never notifies it.  The hook clears
 * itself after that call.
 * what = 2 (checked builds only, else PURLIN_ERR_UNSUPPORTED): the NEXT
 * zero-staging call on h that runs the vector kernels gets its first segment's
 * destination moved one output extent too far, so that its kernel meets
 * addresses outside the call's buffers; the checked kernel skips every such
 * access and records PURLIN_ERR_BOUNDS.  Test it on outputs that have room
 * behind them (the would-be writes stay inside the caller's allocation).
 * what = 3 (checked builds only): the same with the first segment's sources
 * moved one input extent too far (the largest input extent for a sum); the
 * skipped loads read as zeros.  Test it on inputs with room behind them.
 * what = 0 clears the hook.  Other values: PURLIN_ERR_INVALID_ARG. */
PURLIN_API purlin_status_t purlin_debug_inject(purlin_handle_t h, int what);

/* 1 if this library is the checked build: every global access of its kernels
 * is tested against the call's buffers (inputs, outputs, staging ring) before
 * it is made; an access outside them is skipped and reported as
 * PURLIN_ERR_BOUNDS by purlin_query_status.  0 for the product build.  The
 * checked build is for tests; it is slower. */
PURLIN_API int purlin_debug_checked(void);

/* The first address outside the call's buffers that a checked kernel on h met
 * since the last call of this function (0: none), written to *address; the
 * record is then cleared.  Product builds always report 0.  Synchronizes the
 * device.  Errors: PURLIN_ERR_INVALID_ARG (NULL), PURLIN_ERR_CUDA. */
PURLIN_API purlin_status_t purlin_debug_violation(purlin_handle_t h, uint64_t* address);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_DEBUG_H */
