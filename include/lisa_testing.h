/*
 * lisa_testing.h -- test hooks of liblisa.so.  Not part of the layer's
 * supported interface: these entry points let a test exercise the library's
 * failure reporting without faulting or hanging a GPU, and reach a forward
 * kernel that lisa_forward does not choose.
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

/*
 * The LiSA forward (the layer of lisa_forward: same arguments, layouts,
 * ownership, workspace size and error codes) through the single-kernel
 * tensor-core path: one thread-block cluster per (batch, head) slice keeps
 * that slice's K, its statistics and its local-branch results on chip and
 * reads Q, K and V from device memory once.  It serves bf16 layers with
 * d_h = d_v = 64, walk weights shared by all tokens (LISA_W_FIXED,
 * LISA_W_GEOMETRIC, or T = 0), the ReLU or identity feature map, an even
 * number of grid rows and 8..64 columns in steps of 8 whose slice fits the
 * cluster's shared memory; any other layer returns LISA_ERR_UNSUPPORTED with
 * nothing launched.  lisa_forward runs the two-kernel chain instead, which
 * measured faster on every layer this path serves (the 56 x 56 PVT stage:
 * 31.8 against 35.3 us at T = 3); this entry point keeps the single kernel
 * tested.  Asynchronous on `stream`.
 */
lisa_status lisa_forward_resident(const void *Q, const void *K, const void *V, void *O, int B,
                                  int heads, int H, int W, int d_h, int d_v, int T,
                                  const lisa_weights *wts, const float *alpha, float eps,
                                  int relu_inputs, int dtype, void *workspace,
                                  size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LISA_TESTING_H_ */
