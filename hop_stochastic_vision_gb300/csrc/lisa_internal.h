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
    int T;             // truncation depth (2 for the untruncated walk: w_0 V + Q~ U-bar)
    int untruncated;   // geometric walk without truncation: U-bar = beta (1-beta) (I - beta M)^-1 U_1
    float beta;        // its continue probability
    int relu;          // feature map of Q and K on load: 0 none, 1 ReLU, 2 ELU + 1 (SIMT chains only)
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

    int family;          // kFamilySimt / kFamilyTc
    int resident;        // 1: the single-kernel tensor-core forward (test entry point only)
    int tc_split;        // 1: the tensor-core split chain even where the fused one fits
    int k_raw;           // 1: the statistics' K operand takes no feature map (another tensor stands in for K)

    // workspace views
    int *err;        // error word (bounded device waits that gave up)
    float *s_part;   // [slices][C][D]        partial sum_j K_j
    // SIMT family
    float *u_part;   // [slices][C][D][D]     partial K^T V
    float *m_part;   // [slices][C][D][D]     partial K^T Q~
    float *s_red;    // [slices][D]           sum_j K_j
    float *ucat;     // [slices][max(T-1,1)][D][D]  U_1..U_(T-1), or [slices][D][D] folded
    // tensor-core family
    int tc_cluster;        // CTAs per cluster in the stats kernel (divides chunks)
    float *tc_part;        // [slices][chunks / cluster][128][64] cluster-reduced [U_1^T ; M^T]
    uint8_t *tc_bepi;      // [slices][64 * n_umat + 16][128 B] bf16 epilogue operand
    uint8_t *tc_w1img;     // [2][64][128 B] bf16 MLP first-layer weights
};

// Bits of the workspace's error word (the first int of every forward
// workspace): a bounded device wait that gave up.  The first kernel of each
// forward chain clears the word; lisa_query_status reads it.
constexpr int kErrTimeoutLoad = 1;   // a wait for a TMA load or a peer's data
constexpr int kErrTimeoutMma = 2;    // a wait for a tensor-core product or a buffer release

// Test hook: one CTA waits, with a limit of `cycles` SM cycles, on an
// mbarrier that nothing arrives on, through the same bounded wait the
// tensor-core kernels use, and records kErrTimeoutLoad in *err when the wait
// gives up (it clears *err first).
cudaError_t launch_wait_selftest(int *err, long long cycles, cudaStream_t stream);

constexpr int kFamilySimt = 0;
constexpr int kFamilyTc = 1;

struct Plan {
    int family;
    int chunks, chunk, cluster;
    size_t off_err, off_s_part, off_u_part, off_m_part, off_s_red, off_ucat;
    size_t off_tc_part, off_tc_bepi, off_tc_w1img;
    size_t total;
};

// Which kernel family serves a problem: the tensor-core chain for bf16 with
// d = 64 (when its TMEM budget holds), the SIMT chain otherwise.
int choose_family(int dtype, int D, int T, int wmode, int hidden);

// Deterministic split-K plan and workspace carve-up; the same function serves
// lisa_workspace_bytes and lisa_forward, so the two always agree.
Plan make_plan(int slices, int n, int D, int T, int dtype, int wmode, int hidden);

// Kernel families.  Each launches its kernels in order on `stream`; with
// stage >= 0 it launches only that one (for per-kernel timing).  Returns
// cudaSuccess or the first launch error.
constexpr int kSimtStages = 4;
extern const char *const kSimtStageNames[kSimtStages];
cudaError_t launch_simt(const Problem &p, cudaStream_t stream, int stage);

cudaError_t launch_tc(const Problem &p, cudaStream_t stream, int stage);
// The tensor-core split chain's first two kernels only: the key-sum partials
// (s_part, one per chunk) and the cluster-reduced [U_1^T ; M^T] partials
// (tc_part, [slices][chunks / cluster][128][64] fp32), for a caller that
// reduces them itself.  Without the key sum, the statistics kernel alone
// reuses the s_part an earlier call left.
cudaError_t launch_tc_stats_partials(const Problem &p, cudaStream_t stream, bool with_keysum = true);
// The single-kernel tensor-core forward (one thread-block cluster per slice,
// K resident in shared memory): bf16, d = 64, weights shared by all tokens
// (truncated or untruncated walk), ReLU or no feature map, grids with an even
// number of rows and 8 to 64 columns in steps of 8, when its shared-memory
// plan fits.
bool tc_resident_applies(int slices, int H, int W, int D, int dtype, int wmode, int untruncated, int relu);
cudaError_t launch_tc_resident(const Problem &p, cudaStream_t stream);
// The tensor-core chain is 2 kernels when a slice's chunks fit one cluster
// (fused statistics), else 4.
int tc_num_stages(int chunks, int cluster, int chunk);
const char *tc_stage_name(int chunks, int cluster, int chunk, int stage);

}  // namespace lisa
