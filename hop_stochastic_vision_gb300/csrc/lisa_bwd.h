// lisa_bwd.h -- host-side problem of one lisa_backward call and its
// launcher.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "lisa_internal.h"

namespace lisa {

// One lisa_backward call: the forward's problem (sizes, weights, inputs and
// the statistics partials the forward's SIMT kernels fill) plus the
// upstream gradient, the outputs and the backward's workspace views.
struct BwdProblem {
    Problem fwd;
    // bf16, d = 64, ReLU or no feature map: the statistics come from the
    // tensor-core split chain (tcfwd's workspace views) instead of the SIMT one
    int tc_stats;
    Problem tcfwd;
    // with tc_stats, fixed truncated walk: dUbar's partials from the same
    // kernel (dO standing in for V and K): rows 64 + a of each part are
    // (Q~^T dO)[a][.], [S][parts][128][64]
    int tc_dub;
    float *tcdub;
    const void *dO;
    void *dQ, *dK, *dV;
    float *dalpha;       // device [heads], overwritten
    int tpb, nblk;       // tokens per block of the per-token kernels; blocks per slice
    int ntile;           // 8 x 8 tiles per slice of the tiled token pass (0: 32-token blocks throughout)
    int nh;              // stored U_k matrices: max(T - 1, 1)
    float *Mred;         // [S][D][D]      M = K^T Q~
    float *Uk;           // [S][nh][D][D]  U_1 .. U_(T-1) (untruncated: Z), transposed
    float *Ubar;         // [S][D][D]
    float *UbarT;        // [S][D][D]      Ubar transposed
    float *dub_part;     // [S][C][D][D]   partial dUbar
    float *lstat;        // [S][n][4]      window softmax max, sum, dl_i . l_i
    float *dal_part;     // [S][nblk]
    float *ds_part;      // [S][nblk][D]
    float *dM, *dU1;     // [S][D][D]
    float *dMT, *dU1T;   // [S][D][D]      the same, transposed
    uint16_t *bimg;      // [S][5 D][D] bf16: [alpha Ubar^T; dM; dU_1^T; dM^T; dU_1] (bf16, d = 64)
    uint16_t *ubimg;     // [S][2][D][D] bf16: Ubar row-major as hi and lo terms (hi + lo ~ Ubar)
    float *ds_red;       // [S][D]
    float *dal_slice;    // [S]
    float *dk_part;      // [S][n][D]      dK without ds, fp32
    // adaptive (MLP) walk weights only (null otherwise)
    float *Ukn;          // [S][nh][D][D]  U_1 .. U_(T-1), row-major (the SIMT adaptive-weight pass)
    uint16_t *ukimg;     // [S][nh][2][64][72] bf16: U_k rows as hi, lo terms (72-wide rows; bf16, d = 64)
    uint16_t *w1img;     // [2][64][136] bf16: W1 rows as hi, lo terms (136-wide rows; bf16, d = 64)
    uint16_t *ukimgT;    // [S][nh][64][72] bf16: alpha U_k^T, row c, column a (72-wide rows; bf16, d = 64)
    float *wtok;         // [S][n][T]      per-token walk weights w_i
    float *dzbuf;        // [S][n][T]      dL/dz_i (softmax logits)
    float *hbuf;         // [S][n][hid]    h_i = GELU(W1 x_i + b1)
    float *dabuf;        // [S][n][hid]    dL/d(W1 x_i + b1)
    float *dxm;          // [S][n][2 D]    the MLP's share of dL/dq_i, dL/dk_i
    float *dukp;         // [S][C][T-1][D][D]  partial dU_k = sum_i w_ik Q~_i^T dg_i
    float *pw1, *pb1, *pw2, *pb2;   // [S][C][...] partial parameter gradients
    float *dW1, *db1, *dW2, *db2;   // caller's outputs
    int mlp;             // adaptive weights: the fields above are set
};

cudaError_t launch_bwd(const BwdProblem &b, cudaStream_t stream);

}  // namespace lisa
