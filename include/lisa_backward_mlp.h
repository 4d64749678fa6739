/*
 * lisa_backward_mlp.h -- C ABI of the LiSA backward pass with the adaptive
 * (MLP) walk weights, liblisa.so.
 *
 * With LISA_W_MLP every token i draws its own walk weights,
 * w_i = softmax(W2 GELU(W1 [q_i; k_i] + b1) + b2) over the T walk lengths
 * ("LiSA: Linear Stochastic Attention for Long-Range Visual Modeling",
 * reading note §2.4; paper Eq. 10, Supp. Sec. 8), so the backward has two
 * more parts than lisa_backward's (include/lisa.h): the gradient through the
 * per-token weights into q_i and k_i, and the gradients of the MLP's
 * parameters, which every head and batch element shares.
 *
 * Conventions, checks, statuses and stream behaviour are those of
 * lisa_backward in include/lisa.h.  Arithmetic as there; for bf16 at d = 64
 * with ReLU or no feature map the MLP's contractions run on the tensor cores
 * too (W1, U_k and the hidden-layer gradients enter as bf16 hi + lo terms,
 * fp32 accumulation), and GELU and its derivative take erf from
 * Abramowitz & Stegun 7.1.26 (absolute error <= 1.5e-7), as the forward's
 * adaptive-weight path does.
 */
#ifndef LISA_BACKWARD_MLP_H_
#define LISA_BACKWARD_MLP_H_

#include "lisa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The MLP parameters' gradients: device fp32 buffers, written (not
 * accumulated), summed over every (batch, head) slice; the shapes of
 * lisa_weights' W1, b1, W2, b2. */
typedef struct lisa_mlp_grads {
    float *dW1;   /* [hidden][2*d_h] */
    float *db1;   /* [hidden] */
    float *dW2;   /* [T][hidden] */
    float *db2;   /* [T] */
} lisa_mlp_grads;

/* Bytes of device workspace lisa_backward_mlp needs (a host computation;
 * 0 for arguments it would reject).  hidden: the MLP's width. */
size_t lisa_backward_mlp_workspace_bytes(int B, int heads, int H, int W, int d_h, int d_v, int T,
                                         int hidden, int dtype);

/*
 * Gradients of the layer with adaptive weights (wts->mode == LISA_W_MLP,
 * 1 <= T <= LISA_MAX_T_MLP, 1 <= hidden <= LISA_MAX_HIDDEN) for the upstream
 * gradient dO: dQ, dK, dV, dalpha as lisa_backward writes them, and the MLP
 * parameters' gradients into *mgrads.  Any other weight mode, or a missing
 * mgrads buffer, returns LISA_ERR_INVALID_ARG.
 */
lisa_status lisa_backward_mlp(const void *Q, const void *K, const void *V, const void *dO, void *dQ,
                              void *dK, void *dV, float *dalpha, const lisa_mlp_grads *mgrads,
                              int B, int heads, int H, int W, int d_h, int d_v, int T,
                              const lisa_weights *wts, const float *alpha, float eps,
                              int relu_inputs, int dtype, void *workspace, size_t workspace_bytes,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LISA_BACKWARD_MLP_H_ */
