/*
 * lisa.h -- C ABI of the GB300 (sm_103a) LiSA forward layer library, liblisa.so.
 *
 * LiSA ("LiSA: Linear Stochastic Attention for Long-Range Visual Modeling",
 * arXiv 2611.04216v2; cited from its reading note, sections 2.1-2.5) works
 * per (batch, head) slice on an H x W token grid, n = H*W tokens:
 *
 *   feature map      Q = ReLU(Xq), K = ReLU(Xk)                 [note §2.1]
 *   transition       Q~_i = Q_i / (Q_i . sum_j K_j + eps),
 *                    S = Q~ K^T  (row-stochastic, never formed)  [note §2.2]
 *   global branch    g_i = sum_{k<T} w_k(i) (S^k V)_i, evaluated as
 *                    S^k V = Q~ U_k, U_1 = K^T V, U_k = (K^T Q~) U_(k-1)
 *                                                   [note §2.3; paper Eq. 8]
 *   walk weights     geometric w_k = (1-beta) beta^k / (1-beta^T)
 *                                                   [note §2.2; paper Eq. 4]
 *                    or, untruncated (T = 0), (1-beta) beta^k for every
 *                    k >= 0: g = (1-beta) (I - beta S)^-1 V  [note §2.3, the
 *                    closing remark on the geometric series]
 *                    or per token and head: softmax(W2 GELU(W1 [q_i;k_i] + b1) + b2)
 *                                          [note §2.4; paper Eq. 10, Supp. 8]
 *   local branch     softmax over the token and its in-grid 8-neighbours of
 *                    q_i . k_j / sqrt(d_h), applied to V   [note §2.4]
 *   output           o_i = alpha_h g_i + (1 - alpha_h) l_i  [note §2.4; Fig. 2]
 *
 * Conventions shared by every entry point:
 *   - Tensors are contiguous row-major: Q, K [B][heads][H*W][d_h] and
 *     V, O [B][heads][H*W][d_v]; token index i = r*W + c.
 *   - dtype LISA_F32: fp32 in, fp32 out, fp32 arithmetic throughout.
 *     dtype LISA_BF16: bf16 in, bf16 out (round to nearest even), fp32
 *     accumulation; bf16 tensor-core operands where the contraction allows.
 *   - d_h == d_v, each one of 16, 32, 64; other sizes give LISA_ERR_UNSUPPORTED
 *     (the layer widths of every configuration here have d_v = d_h; d_v != d_h
 *     is rejected rather than served).
 *   - Device pointers must be 16-byte aligned.  O must not overlap an input.
 *   - The library allocates no device memory: the caller owns every buffer,
 *     including the workspace.  Its host-side state is limited to lookups
 *     cached once per device (the kernels' shared-memory limits, the tensor
 *     map encoder, the no-alloc scratch address below), and its one device
 *     buffer is that scratch array of lisa_forward_noalloc.  Calls on
 *     different streams with different workspaces may run concurrently.
 *   - Every argument is checked on the host before anything is launched; a
 *     bad argument returns its status and launches nothing.  Launch
 *     failures return LISA_ERR_CUDA.  The call is asynchronous on `stream`
 *     (a cudaStream_t; NULL = legacy default stream) and never synchronises.
 */
#ifndef LISA_H_
#define LISA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lisa_status {
    LISA_OK = 0,
    LISA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, T < 1, beta outside [0,1), eps <= 0, misalignment */
    LISA_ERR_UNSUPPORTED = 2,  /* d_h / d_v / T / hidden outside what the kernels are built for */
    LISA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than lisa_workspace_bytes() */
    LISA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    LISA_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up */
} lisa_status;

typedef enum lisa_dtype { LISA_F32 = 0, LISA_BF16 = 1 } lisa_dtype;

/* Walk-weight modes [note §2.2, §2.4]. */
typedef enum lisa_wmode {
    LISA_W_GEOMETRIC = 0,  /* w_k = (1-beta) beta^k / (1-beta^T), computed on the host in double */
    LISA_W_FIXED = 1,      /* w[0..T-1] given by the caller (host memory), any real values */
    LISA_W_MLP = 2         /* per-token, per-head weights from the 2-layer MLP + softmax */
} lisa_wmode;

#define LISA_MAX_T 16        /* largest truncation depth T */
#define LISA_MAX_T_MLP 8     /* largest T with adaptive (MLP) weights */
#define LISA_MAX_HIDDEN 64   /* largest MLP hidden width */

typedef struct lisa_weights {
    int mode;          /* lisa_wmode */
    float beta;        /* GEOMETRIC: continue probability, 0 <= beta < 1 */
    const float *w;    /* FIXED: host array [T] */
    const float *W1;   /* MLP: device fp32 [hidden][2*d_h]; input is concat(q_i, k_i) post-ReLU */
    const float *b1;   /* MLP: device fp32 [hidden] */
    const float *W2;   /* MLP: device fp32 [T][hidden] */
    const float *b2;   /* MLP: device fp32 [T] */
    int hidden;        /* MLP: hidden width, 1..LISA_MAX_HIDDEN (32 in the paper's setting) */
} lisa_weights;

/*
 * Bytes of device workspace lisa_forward needs for this problem (a pure
 * host computation; no CUDA call).  Returns 0 for arguments lisa_forward
 * would reject.  The workspace holds the split-K partial sums of sum_j K_j,
 * K^T V and K^T Q~ [note §2.3], the reduced statistics and U_1..U_(T-1).
 * Its first 4 bytes are the call's error word: the first kernel of every
 * forward sets it to 0 and a bounded device wait that gives up sets bits in
 * it (lisa_query_status reads it).  Every other byte is written by the call
 * before it is read, so the buffer needs no initialisation.
 * T = 0 (the untruncated walk) is accepted and sized like T = 2.
 */
size_t lisa_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                            int dtype);

/*
 * The LiSA forward layer [note §2.1-2.4] on device buffers.
 *   Q, K        device [B][heads][H*W][d_h], dtype; raw projections Xq, Xk
 *               when relu_inputs = 1 (ReLU applied on load) or 2 (the
 *               ELU(x) + 1 feature map applied on load [note §2.1; paper
 *               Table 8]; served by the SIMT kernels for every dtype), or
 *               already feature-mapped (non-negative) when relu_inputs = 0.
 *   V           device [B][heads][H*W][d_v], dtype.
 *   O           device [B][heads][H*W][d_v], dtype; written.
 *   T           truncation depth, 1..LISA_MAX_T (1..LISA_MAX_T_MLP for MLP);
 *               0 with LISA_W_GEOMETRIC: the untruncated walk,
 *               g = (1-beta) (I - beta S)^-1 V.  The library evaluates it as
 *               g = (1-beta) (V + beta Q~ X) with (I - beta M) X = U_1,
 *               M = K^T Q~ (the push-through identity; a d x d solve per
 *               slice).  That system is well posed because the features
 *               are non-negative (relu_inputs = 1 or 2, or inputs that already
 *               are): I - beta M is then a nonsingular M-matrix.  T = 0 with
 *               LISA_W_FIXED or LISA_W_MLP is LISA_ERR_INVALID_ARG.
 *   wts         host struct; see lisa_weights.
 *   alpha       device fp32 [heads]: branch mix per head, used as given.
 *   eps         stabiliser of the row normaliser, > 0 (the paper's setting: 1e-6).
 *   workspace   device, >= lisa_workspace_bytes(...) bytes, 16-byte aligned.
 *   stream      cudaStream_t.
 */
lisa_status lisa_forward(const void *Q, const void *K, const void *V, void *O, int B,
                         int heads, int H, int W, int d_h, int d_v, int T,
                         const lisa_weights *wts, const float *alpha, float eps,
                         int relu_inputs, int dtype, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * End-to-end variant on host buffers: copies hQ, hK, hV (host, ideally
 * pinned) into the caller's device buffers dQ, dK, dV, runs lisa_forward,
 * and copies dO back into hO, all enqueued on `stream` in that order.  The
 * host buffers must stay valid until the stream has drained; the call does
 * not wait for it.  Sizes and the other arguments are as for lisa_forward.
 */
lisa_status lisa_forward_host(const void *hQ, const void *hK, const void *hV, void *hO,
                              void *dQ, void *dK, void *dV, void *dO, int B, int heads,
                              int H, int W, int d_h, int d_v, int T,
                              const lisa_weights *wts, const float *alpha, float eps,
                              int relu_inputs, int dtype, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Per-kernel access for profiling.  One lisa_forward call is a fixed chain of
 * lisa_num_stages(...) kernel launches; lisa_forward_stage(i, ...) launches
 * only kernel i of that chain with the same arguments and checks.  Running
 * stages 0 .. n-1 in order on one stream with one workspace computes exactly
 * what lisa_forward computes (each stage reads what the earlier ones left in
 * the workspace), so a caller can put timing events between the kernels.
 * The chain depends on the problem's sizes, dtype and weights (mode, MLP
 * width); lisa_num_stages returns 0 for arguments lisa_forward would reject
 * or for an empty problem.  lisa_stage_name returns the kernel's name, or
 * NULL for a bad index.
 * A bad stage index, or relu_inputs = 2 (the list describes the chains of
 * relu_inputs 0 and 1), returns LISA_ERR_INVALID_ARG.
 */
int lisa_num_stages(int B, int heads, int H, int W, int d_h, int T, int dtype,
                    const lisa_weights *wts);
const char *lisa_stage_name(int B, int heads, int H, int W, int d_h, int T, int dtype,
                            const lisa_weights *wts, int stage);
lisa_status lisa_forward_stage(int stage, const void *Q, const void *K, const void *V, void *O,
                               int B, int heads, int H, int W, int d_h, int d_v, int T,
                               const lisa_weights *wts, const float *alpha, float eps,
                               int relu_inputs, int dtype, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * lisa_forward without a workspace argument, for callers that cannot
 * allocate device memory when they run the layer: an operator inside an
 * inference engine or framework that owns all device memory through its own
 * pool, planned before execution, so the operator may not call cudaMalloc;
 * or a latency-bound serving loop that cannot take the device-wide
 * synchronisation a cudaFree implies.  The paper has no counterpart; this is
 * a property of the library, not of the method.
 *
 * Instead of a caller workspace it uses one scratch array compiled into the
 * library: LISA_NOALLOC_SCRATCH_BYTES of device memory on every GPU that
 * loads liblisa.so, held until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - The call's own workspace need (what lisa_forward would use for these
 *     sizes, weight mode and feature map, at most lisa_workspace_bytes(...))
 *     must fit in LISA_NOALLOC_SCRATCH_BYTES; a larger problem is rejected
 *     with LISA_ERR_WORKSPACE before anything is launched.  Use lisa_forward
 *     with your own workspace there.
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process.  Make that first call before any stream capture
 *     begins.  Later calls do no runtime lookups.  Call with the device of
 *     `stream` current.  Calls must not cross a cudaDeviceReset (or any
 *     other reset of the device's primary context): the kept address would
 *     be stale afterwards.
 *   - Every call on a device shares the one array, and it keeps whatever the
 *     last call left there.  The only entry that must start at zero, the
 *     error word, is cleared by each call's first kernel; every other entry
 *     is written before it is read.  Calls whose kernels overlap on the GPU
 *     (different streams, no ordering between them) race on the array and
 *     give wrong results: order them on one stream, or give each its own
 *     workspace through lisa_forward.
 *   - A timed-out device wait cannot be queried for these calls (the scratch
 *     array's address is not handed out); lisa_query_status serves
 *     lisa_forward's caller-owned workspaces.
 * Other arguments, checks and statuses are those of lisa_forward.
 */
#define LISA_NOALLOC_SCRATCH_BYTES (32u << 20)
lisa_status lisa_forward_noalloc(const void *Q, const void *K, const void *V, void *O, int B,
                                 int heads, int H, int W, int d_h, int d_v, int T,
                                 const lisa_weights *wts, const float *alpha, float eps,
                                 int relu_inputs, int dtype, void *stream);

/*
 * Backward pass of the layer: the gradients of a loss L with respect to the
 * layer's inputs, given dO = dL/dO (the chain rule through the forward
 * above; the paper trains LiSA backbones end to end [note §3]).
 *   Q, K, V     the forward's inputs (device, dtype, [B][heads][H*W][d]).
 *   dO          device [B][heads][H*W][d_v], dtype: upstream gradient.
 *   dQ, dK, dV  device, dtype, same shapes; written: dL/dQ, dL/dK, dL/dV
 *               of the raw inputs (through the feature map: relu_inputs = 1
 *               zero where the input is <= 0; 2 scaled by exp(x) there).
 *   dalpha      device fp32 [heads]; written (not accumulated): dL/dalpha_h,
 *               summed over the batch.
 * Weights: LISA_W_GEOMETRIC (T >= 1, or T = 0 untruncated) and LISA_W_FIXED;
 * LISA_W_MLP returns LISA_ERR_UNSUPPORTED.  Outputs may not overlap each
 * other or any input.  Arithmetic is fp32 (bf16 inputs widened, bf16
 * outputs rounded to nearest even), except that for bf16 at d = 64 with
 * ReLU or no feature map the contractions run on the tensor cores with bf16
 * operands (Q~, the window weights, the d x d matrices) and fp32
 * accumulation; every sum runs in a fixed order, so the result is the same
 * on every run.  The workspace (>= the bytes
 * lisa_backward_workspace_bytes returns, 16-byte aligned) needs no
 * initialisation.  Checks, statuses and stream behaviour as for
 * lisa_forward, with one addition: on the tensor-core path the call forks
 * one statistics launch onto a library-owned stream of the current device
 * and joins it back into `stream` before its last kernel, so all of its work
 * stays ordered after earlier work on `stream` and before later work (and a
 * CUDA graph captured from `stream` holds the fork and the join).  That
 * stream is created by the first such call that is not made during stream
 * capture; until then the launch runs on `stream` itself.  An empty problem
 * (B * heads * H * W == 0) only zeroes dalpha.
 */
size_t lisa_backward_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                                     int dtype);
lisa_status lisa_backward(const void *Q, const void *K, const void *V, const void *dO, void *dQ,
                          void *dK, void *dV, float *dalpha, int B, int heads, int H, int W,
                          int d_h, int d_v, int T, const lisa_weights *wts, const float *alpha,
                          float eps, int relu_inputs, int dtype, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Failure reporting of the device side.  The tensor-core kernels bound every
 * wait (on a TMA load, a tensor-core product, a buffer release, a peer's
 * data) to about one second; a wait that gives up sets a bit in the error
 * word at the start of the call's workspace and the kernel finishes along
 * its normal path (every CTA still frees its tensor memory and drains its
 * bulk stores), leaving the outputs undefined.  The backward's tensor-core
 * kernels do the same in the backward workspace.  lisa_forward and
 * lisa_backward return before the kernels run, so they cannot see this.
 * lisa_query_status reads the word of `workspace` (the one passed to the
 * last lisa_forward or lisa_backward call on it) after the work queued on
 * `stream` has finished: it synchronises `stream` and returns
 * LISA_ERR_TIMEOUT if any wait gave up, LISA_OK otherwise, or LISA_ERR_CUDA
 * if the read itself failed.  A null or misaligned workspace is
 * LISA_ERR_INVALID_ARG.  The next call on the workspace clears the word
 * again.
 */
lisa_status lisa_query_status(const void *workspace, void *stream);

/* Static, human-readable name of a status code. */
const char *lisa_status_string(int status);

/* ABI version, bumped on any signature change: major * 100 + minor. */
int lisa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LISA_H_ */
