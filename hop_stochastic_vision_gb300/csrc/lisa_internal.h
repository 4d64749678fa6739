// lisa_internal.h -- host-side plan of one lisa_forward call and the launcher
// entry points of the kernel families.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "lisa.h"

namespace lisa {

// Everything a kernel family needs for one call: problem sizes, the weights
// already resolved on the host, and views into the caller's workspace.
struct Problem {
    const void *Q, *K, *V;
    void *O;
    int slices;        // B * heads
    int heads;
    int H, W, n;       // grid and tokens per slice
    int D;             // d_h = d_v
    int T;             // truncation depth
    int relu;          // apply ReLU to Q and K on load
    float eps;
    const float *alpha;  // device [heads]
    int wmode;           // LISA_W_* after GEOMETRIC has been resolved to FIXED
    float w[LISA_MAX_T]; // FIXED / GEOMETRIC walk weights (fp32 of the double values)
    const float *W1, *b1, *W2, *b2;  // MLP (device)
    int hidden;
    int dtype;           // LISA_F32 / LISA_BF16

    // split-K plan over the tokens of a slice
    int chunks;          // C: chunks per slice
    int chunk;           // tokens per chunk (last one may be shorter)

    // workspace views (fp32)
    float *s_part;   // [slices][C][D]        partial sum_j K_j
    float *u_part;   // [slices][C][D][D]     partial K^T V
    float *m_part;   // [slices][C][D][D]     partial K^T Q~
    float *s_red;    // [slices][D]           sum_j K_j
    float *ucat;     // [slices][max(T-1,1)][D][D]  U_1..U_(T-1), or [slices][D][D] folded
    void *aux;       // [slices][...] kernel-family specific (bf16 operand copies)
};

struct Plan {
    int chunks, chunk;
    size_t off_s_part, off_u_part, off_m_part, off_s_red, off_ucat, off_aux;
    size_t total;
};

// Deterministic split-K plan and workspace carve-up; the same function serves
// lisa_workspace_bytes and lisa_forward, so the two always agree.
Plan make_plan(int slices, int n, int D, int T, int dtype);

// Kernel families.  Each launches its kernels in order on `stream`; with
// stage >= 0 it launches only that one (for per-kernel timing).  Returns
// cudaSuccess or the first launch error.
constexpr int kSimtStages = 4;
extern const char *const kSimtStageNames[kSimtStages];
cudaError_t launch_simt(const Problem &p, cudaStream_t stream, int stage);

}  // namespace lisa
