/*
 * gdn_testing.h -- test hooks of the GDN library. Not part of the layer API: the method has no
 * counterpart, and nothing in the layer calls these.
 *
 * Every wait of the kernels on an asynchronous copy or tensor-core group is bounded; when one
 * runs out the kernel sets GDN_DEVERR_TIMEOUT in the caller's error word and stops the work
 * that needed it, leaving the context usable. These hooks make one such wait run out on the
 * GPU (a barrier that nothing arrives on, waited for with a 10 ms bound), so that the failure
 * path and its error reporting can be tested without faulting or hanging anything.
 */
#ifndef GDN_TESTING_H
#define GDN_TESTING_H

#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Test fault modes. */
#define GDN_TEST_FAULT_NONE 0
/* The persistent decode kernel (batches with at least half as many (row, k-head) units as the
 * GPU has SMs, ungated or gated): its first consumer warp of CTA 0 leaves at its first wait.
 * The other waits of that CTA then run out in turn (about a second each) and every role stops;
 * the call's outputs and the states of its active slots are not to be trusted, and slots it
 * does not address are untouched. */
#define GDN_TEST_FAULT_DECODE_CONSUMER 1
/* The tensor-core state pass of the chunked prefill (dk = dv = 128): compute warp 0 of its
 * first CTA gives up its first group-2 wait. The warps of that CTA leave the chunk loop
 * together, drain their bulk copies and MMA groups and free tensor memory; that CTA's
 * sequence and value head get no final state, every other one is computed as usual. */
#define GDN_TEST_FAULT_PREFILL_PASS 2

/*
 * gdn_testing_set_fault -- sets the fault mode of every kernel launched from now on, on the
 * current device (a synchronous copy to a device flag); GDN_TEST_FAULT_NONE restores normal
 * operation. Returns GDN_ERR_INVALID_ARG for an unknown mode, GDN_ERR_CUDA if the copy fails.
 */
gdn_status gdn_testing_set_fault(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */
