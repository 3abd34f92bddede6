/*
 * purlin_debug.h -- fault injection for testing the bounded waits.
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

#include "purlin.h"

#ifdef __cplusplus
extern "C" {
#endif

/* what = 1: in the NEXT staged (PURLIN_VARIANT_STAGED) call on h, the producer
 * of channel 0 stages its first chunk but never notifies it.  The hook clears
 * itself after that call.  what = 0 clears it.  Other values:
 * PURLIN_ERR_INVALID_ARG. */
PURLIN_API purlin_status_t purlin_debug_inject(purlin_handle_t h, int what);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_DEBUG_H */
