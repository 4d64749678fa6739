/*
 * lisa_testing.h -- test hooks of liblisa.so.  Not part of the layer: these
 * entry points exist so that a test can exercise the library's failure
 * reporting without faulting or hanging a GPU.
 */
#ifndef LISA_TESTING_H_
#define LISA_TESTING_H_

#include <stddef.h>

#include "lisa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs, on `stream`, one thread block that clears the error word at the start
 * of `workspace` (device, 16-byte aligned, >= 4 bytes) and then waits on an
 * mbarrier that nothing ever arrives on, with a limit of `cycles` SM cycles,
 * through the same bounded wait the tensor-core kernels use.  When the limit
 * runs out the block records a timeout in the error word and exits; nothing
 * else is in flight, so the context stays usable.  lisa_query_status on the
 * same workspace then returns LISA_ERR_TIMEOUT.  cycles < 0, a null or
 * misaligned workspace, or fewer than 4 bytes: LISA_ERR_INVALID_ARG, nothing
 * launched.  Asynchronous on `stream`.
 */
lisa_status lisa_selftest_wait_timeout(long long cycles, void *workspace, size_t workspace_bytes,
                                       void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LISA_TESTING_H_ */
