/*
 * pa_testing.h -- a test hook of libpa.so, outside the attention ABI of pa.h.
 *
 * Every wait in the kernels is bounded: a role that waits on another role's
 * progress (a copy to land, a score tile, a free ring slot) gives up after a
 * cycle limit, records PA_STATUS_BIT_TIMEOUT, still lets the copies and
 * tensor-core operations it issued finish, frees its tensor memory and exits,
 * so that the context stays usable and pa_status_read reports
 * PA_ERR_TIMEOUT. The limit is about two seconds, so a healthy launch never
 * meets it; this call lowers it so that a test can make those waits run out
 * on a correct launch and check the path. Not for production use.
 */
#ifndef PA_TESTING_H
#define PA_TESTING_H

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_testing_set_wait_limit -- the cycle limit of the decode kernels' waits
 * (the CUDA-core, mma.sync and 64-row tcgen05 kernels), for every later
 * pa_forward / pa_forward_device_plan / pa_forward_noalloc call of the
 * process; 0 restores the default (about two seconds). Under a lowered limit
 * the CUDA-core and mma.sync kernels poll their copies without suspending, so
 * a copy that has not landed within the limit makes the wait run out; the
 * tcgen05 kernel keeps its suspending polls, so there a wait runs out when it
 * outlasts one suspension and the limit (its waits on other roles do). The
 * waits a CTA makes for its own copies and tensor-core operations before it
 * exits keep the default whatever this is, and the prefill kernels always use
 * the default. Returns PA_ERR_INVALID_ARG for a negative value.
 */
pa_status pa_testing_set_wait_limit(long long cycles);

#ifdef __cplusplus
}
#endif
#endif /* PA_TESTING_H */
