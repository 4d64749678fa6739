// lisa_bwd.cu -- backward pass of the LiSA layer (fixed walk weights, incl.
// geometric and the untruncated walk): dL/dXq, dL/dXk, dL/dV, dL/dalpha for
// an upstream gradient dO, every dtype and head width the forward serves:
// fp32 on CUDA cores, and for bf16 at d = 64 the contractions on the tensor
// cores (bf16 operands, fp32 accumulation).
//
// The chain rule through the forward's steps ("LiSA: Linear Stochastic
// Attention for Long-Range Visual Modeling", reading note §2.1-2.4; paper
// Eq. 4, Eq. 8, Sec. 3.2), with dg = alpha dO and dl = (1 - alpha) dO:
//   dalpha = sum_i dO_i . (g_i - l_i)
//   dUbar = Q~^T dg;   G_(T-1) = w_(T-1) dUbar, G_k = w_k dUbar + M^T G_(k+1);
//   dM = sum_{k>=2} G_k U_(k-1)^T, dU_1 = G_1   (untruncated: dU_1 = A^-T dZ,
//   dM = beta (A^-T dZ) Z^T, A = I - beta M, dZ = beta (1-beta) dUbar)
//   dQ~_i = dg_i Ubar^T + dM^T K_i;  c_i = (dQ~_i . Q~_i) / r_i;
//   dQ_i = dQ~_i / r_i - c_i s;  ds = -sum_i c_i Q_i
//   dV_j = w_0 dg_j + dU_1^T K_j;  dK_j = dU_1 V_j + dM Q~_j + ds
//   local window (a = softmax of q_i . k_j / sqrt(d)):  dV_j += sum_i a_ij dl_i,
//   de_ij = a_ij (dl_i . V_j - dl_i . l_i), dQ_i += sum_j de_ij K_j / sqrt(d),
//   dK_j += sum_i de_ij Q_i / sqrt(d)  (the window is symmetric: i in N(j)
//   exactly when j in N(i), so each token gathers its own terms)
//   feature map: dXq = dQ [Xq > 0], dXk = dK [Xk > 0].
//
// Launch chain (after the statistics: the forward's two SIMT kernels, or for
// bf16 at d = 64 without the ELU map the tensor-core split kernels, which
// leave the split-K partials of s, U_1 = K^T V and M = K^T Q~; there a second
// split-statistics launch with dO as its V and K gives dUbar's partials in
// place of step 2, and steps 3 and 5 take a quarter-warp per token):
//   1. bwd_recur      per slice: reduce s, U_1, M; U_k, Ubar (or the solve)
//   2. bwd_stats_dub  per (slice, chunk): partial dUbar = Q~^T (alpha dO)
//   3. bwd_token_a    warp per token: window softmax max / sum, dl_i . l_i,
//                     dalpha terms (per-block partial sums)
//   4. bwd_recur_back per slice: reduce dUbar; G_k; dM, dU_1 (or the solve);
//                     bf16, d = 64, T <= 3: bwd_recur_back_rows, four CTAs per slice
//   5. bwd_token_b    per block of 32 tokens: the d x d products from shared
//                     memory, then a warp per token: dXq, dV, the ds terms
//                     (per-block sums), dK without ds.  bf16, d = 64:
//                     bwd_token_b_tile on 8 x 8 token tiles with their halo in
//                     shared memory, the products and the window on the tensor
//                     cores (B operands from a bf16 image built by bwd_bimg)
//   6. bwd_reduce     per slice: ds and the slice's dalpha
//   7. bwd_finish_k   one thread per element: dXk = (dK + ds) [Xk > 0];
//                     its block 0 also sums dalpha per head over the batch
// With the adaptive (MLP) weights, steps 2-3 become bwd_token_mlp (the
// window statistics, the MLP's forward and backward per token; bf16, d = 64:
// bwd_token_mlp_tc after bwd_mlp_images has built the bf16 U_k and W1 operand
// images) and bwd_stats_duk (one split-K dU_k = sum_i w_ik Q~_i^T dg_i per walk
// length); step 5 adds each token's own walk terms and the MLP's share of
// dq, dk; bwd_mlp_params and bwd_mlp_reduce produce dW1, db1, dW2, db2.
// Every reduction runs in a fixed order: the result does not depend on
// scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "lisa_bwd.h"
#include "lisa_internal.h"
#include "lisa_sm100.cuh"
#include "lisa_solve.cuh"
#include "lisa_tc_common.cuh"

namespace lisa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float *p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
// The feature map applied on load; `fmap` is the call's relu_inputs:
// 0 the inputs are the features, 1 ReLU, 2 ELU(x) + 1.
__device__ __forceinline__ float feature(float x, int fmap) {
    if (fmap == 1) return x < 0.f ? 0.f : x;
    if (fmap == 2) return x > 0.f ? x + 1.f : expf(x);
    return x;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 64 x 64 products in shared memory (row stride 64), register-blocked: thread
// t of 256 owns rows a0 = 4 (t / 16) .. a0 + 3 and columns c0 = 4 (t % 16)
// .. c0 + 3 of the result.  acc += A B, with A(a, e) = A[e][a] when kTransA.
template <bool kTransA>
__device__ __forceinline__ void mm64_acc(const float *A, const float *B, float (&acc)[4][4], int tid) {
    const int a0 = 4 * (tid >> 4), c0 = 4 * (tid & 15);
#pragma unroll 4
    for (int e = 0; e < 64; ++e) {
        float av[4];
        if (kTransA) {
            const float4 t = *reinterpret_cast<const float4 *>(A + e * 64 + a0);
            av[0] = t.x; av[1] = t.y; av[2] = t.z; av[3] = t.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = A[(a0 + i) * 64 + e];
        }
        const float4 bv = *reinterpret_cast<const float4 *>(B + e * 64 + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[i][0] = fmaf(av[i], bv.x, acc[i][0]);
            acc[i][1] = fmaf(av[i], bv.y, acc[i][1]);
            acc[i][2] = fmaf(av[i], bv.z, acc[i][2]);
            acc[i][3] = fmaf(av[i], bv.w, acc[i][3]);
        }
    }
}
// Row i of a thread's 4 x 4 block to/from shared or global memory (16-byte aligned rows).
__device__ __forceinline__ void st_row4(float *dst, const float (&v)[4]) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// ---------------------------------------------------------------------------
// 1. reduce the statistics; U_1 .. U_(T-1) and Ubar = sum_k w_k U_k, or for
// the untruncated walk Z = (I - beta M)^-1 U_1 (kept in U_1's place) and
// Ubar = beta (1-beta) Z.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) bwd_recur(BwdProblem b) {
    constexpr int EPT = D * D / kThreads;
    __shared__ float M[D][D];
    __shared__ float U[D][D];
    __shared__ float Un[D][D];
    const Problem &p = b.fwd;
    const int sl = blockIdx.x, tid = threadIdx.x;
    if (b.tc_stats) {
        // tensor-core partials: per part a [U_1^T ; M^T] block of 2D rows x D
        // columns (row e < D: U_1[.][e]; row D + c: M[.][c]), summed in part order
        const Problem &t = b.tcfwd;
        const int parts = t.chunks / t.tc_cluster;
        const float *tp = t.tc_part + (size_t)sl * parts * 2 * D * D;
        for (int idx = tid; idx < D * D; idx += kThreads) {
            // element (a, r) of U_1 and M: row r, column a of the partials (strided
            // global reads, row-contiguous shared-memory writes)
            const int a = idx / D, r = idx % D;
            float m = 0.f, u = 0.f;
            for (int q = 0; q < parts; ++q) {
                u += tp[(size_t)q * 2 * D * D + r * D + a];
                m += tp[(size_t)q * 2 * D * D + D * D + r * D + a];
            }
            U[a][r] = u;
            M[a][r] = m;
        }
        if (tid < D) {
            float acc = 0.f;
            for (int c = 0; c < t.chunks; ++c) acc += t.s_part[((size_t)sl * t.chunks + c) * D + tid];
            p.s_red[(size_t)sl * D + tid] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < D * D; idx += kThreads) b.Mred[(size_t)sl * D * D + idx] = M[idx / D][idx % D];
    } else {
        for (int idx = tid; idx < D * D; idx += kThreads) {
            float m = 0.f, u = 0.f;
            for (int c = 0; c < p.chunks; ++c) {
                const size_t pc = ((size_t)sl * p.chunks + c) * D * D + idx;
                m += p.m_part[pc];
                u += p.u_part[pc];
            }
            M[idx / D][idx % D] = m;
            U[idx / D][idx % D] = u;
            b.Mred[(size_t)sl * D * D + idx] = m;
        }
        if (tid < D) {
            float acc = 0.f;
            for (int c = 0; c < p.chunks; ++c) acc += p.s_part[((size_t)sl * p.chunks + c) * D + tid];
            p.s_red[(size_t)sl * D + tid] = acc;
        }
    }
    __syncthreads();
    float *Uk = b.Uk + (size_t)sl * b.nh * D * D;   // transposed: Uk[c][a] = U_k[a][c]
    float ub[EPT];
    if (p.untruncated) {
        // A = I - beta M stored by columns in Un, R = U_1 by columns in M
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int a = idx / D, c = idx % D;
            Un[c][a] = (a == c ? 1.f : 0.f) - p.beta * M[a][c];
        }
        __syncthreads();
        for (int idx = tid; idx < D * D; idx += kThreads) M[idx % D][idx / D] = U[idx / D][idx % D];
        __syncthreads();
        solve_walk_system<kWarps, (2 * D + kWarps - 1) / kWarps>(&Un[0][0], D, &M[0][0], D, D, D, &U[0][0], tid);
        for (int idx = tid; idx < D * D; idx += kThreads) U[idx / D][idx % D] = M[idx % D][idx / D];
        __syncthreads();
#pragma unroll
        for (int x = 0; x < EPT; ++x) {
            const int idx = tid + x * kThreads;
            Uk[idx] = U[idx % D][idx / D];
            ub[x] = p.beta * (1.f - p.beta) * U[idx / D][idx % D];
        }
    } else {
#pragma unroll
        for (int x = 0; x < EPT; ++x) {
            const int idx = tid + x * kThreads;
            Uk[(idx % D) * D + idx / D] = U[idx / D][idx % D];
            ub[x] = p.T > 1 ? p.w[1] * U[idx / D][idx % D] : 0.f;
            if (b.mlp) b.Ukn[(size_t)sl * b.nh * D * D + idx] = U[idx / D][idx % D];
        }
        for (int k = 2; k < p.T; ++k) {
            if constexpr (D == 64) {   // register-blocked product
                float acc[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
                mm64_acc<false>(&M[0][0], &U[0][0], acc, tid);
                const int a0 = 4 * (tid >> 4), c0 = 4 * (tid & 15);
#pragma unroll
                for (int i = 0; i < 4; ++i) st_row4(&Un[0][0] + (a0 + i) * D + c0, acc[i]);
            } else {
                for (int idx = tid; idx < D * D; idx += kThreads) {
                    const int a = idx / D, e = idx % D;
                    float acc = 0.f;
                    for (int c = 0; c < D; ++c) acc = fmaf(M[a][c], U[c][e], acc);
                    Un[a][e] = acc;
                }
            }
            __syncthreads();
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const float u = Un[idx / D][idx % D];
                U[idx / D][idx % D] = u;
                ub[x] = fmaf(p.w[k], u, ub[x]);
            }
            __syncthreads();
            for (int idx = tid; idx < D * D; idx += kThreads) {
                Uk[(size_t)(k - 1) * D * D + (idx % D) * D + idx / D] = U[idx / D][idx % D];
                if (b.mlp) b.Ukn[((size_t)sl * b.nh + (k - 1)) * D * D + idx] = U[idx / D][idx % D];
            }
        }
    }
#pragma unroll
    for (int x = 0; x < EPT; ++x) {
        const int idx = tid + x * kThreads;
        b.Ubar[(size_t)sl * D * D + idx] = ub[x];
        b.UbarT[(size_t)sl * D * D + (idx % D) * D + idx / D] = ub[x];
        // the bf16 image of Ubar for the tensor-core token pass: hi, then the rest
        const __nv_bfloat16 hi = __float2bfloat16_rn(ub[x]);
        b.ubimg[(size_t)sl * 2 * D * D + idx] = __bfloat16_as_ushort(hi);
        b.ubimg[(size_t)sl * 2 * D * D + D * D + idx] =
            __bfloat16_as_ushort(__float2bfloat16_rn(ub[x] - __bfloat162float(hi)));
    }
}

// ---------------------------------------------------------------------------
// 1' (d = 64, truncated walk, statistics from the tensor-core partials). Step
// 1 split over four CTAs per slice: U_k^T = U_(k-1)^T M^T, so rows e0 .. e0 +
// 15 of every U_k^T (columns of U_k) depend only on the same rows of U_1^T,
// and each CTA carries its 16 rows through the whole recurrence (M^T reduced
// by each).  CTA 0 of a slice also writes s and M.
// ---------------------------------------------------------------------------
constexpr int kRecurSplit = 4;

__global__ void __launch_bounds__(kThreads) bwd_recur_rows(BwdProblem b) {
    constexpr int D = 64, R = D / kRecurSplit;
    __shared__ __align__(16) float Mt[D][D + 4];   // M^T: Mt[c][a] = M[a][c] (padded for the column reads)
    __shared__ __align__(16) float Ut[R][D];   // this CTA's rows of U_k^T
    __shared__ __align__(16) float Un[R][D + 4];   // padded: the last step reads it by columns
    const Problem &p = b.fwd;
    const Problem &t = b.tcfwd;
    const int sl = blockIdx.x / kRecurSplit, cb = blockIdx.x % kRecurSplit, e0 = R * cb, tid = threadIdx.x;
    const int parts = t.chunks / t.tc_cluster;
    const float *tp = t.tc_part + (size_t)sl * parts * 2 * D * D;
    // partials: row e < 64 holds U_1[.][e] (a row of U_1^T), row 64 + c holds M[.][c] (a row of M^T)
    for (int idx = tid; idx < D * D; idx += kThreads) {
        float m = 0.f;
        for (int q = 0; q < parts; ++q) m += tp[(size_t)q * 2 * D * D + D * D + idx];
        Mt[idx / D][idx % D] = m;
    }
    for (int idx = tid; idx < R * D; idx += kThreads) {
        float u = 0.f;
        for (int q = 0; q < parts; ++q) u += tp[(size_t)q * 2 * D * D + e0 * D + idx];
        Ut[idx / D][idx % D] = u;
    }
    if (cb == 0 && tid < D)
        p.s_red[(size_t)sl * D + tid] = sum_partials(t.s_part + (size_t)sl * t.chunks * D, t.chunks, D, tid);
    __syncthreads();
    const size_t so = (size_t)sl * D * D;
    if (cb == 0)
        for (int idx = tid; idx < D * D; idx += kThreads)   // M row-major, rows written whole
            b.Mred[so + idx] = Mt[idx % D][idx / D];
    // thread: row i of the block, columns a0 .. a0 + 3
    const int i = tid >> 4, a0 = 4 * (tid & 15), e = e0 + i;
    float ub[4];
    float *Uk = b.Uk + (size_t)sl * b.nh * D * D;   // transposed: Uk[e][a] = U_k[a][e]
    auto emit = [&](int k) {   // U_k's rows of this thread into the stored copies
        const float4 u = *reinterpret_cast<const float4 *>(&Ut[i][a0]);
        *reinterpret_cast<float4 *>(Uk + (size_t)(k - 1) * D * D + e * D + a0) = u;
        return u;
    };
    {
        const float4 u = emit(1);
        const float w1 = p.T > 1 ? p.w[1] : 0.f;
        ub[0] = w1 * u.x; ub[1] = w1 * u.y; ub[2] = w1 * u.z; ub[3] = w1 * u.w;
    }
    for (int k = 2; k < p.T; ++k) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
            const float x = Ut[i][c];
            const float4 m = *reinterpret_cast<const float4 *>(&Mt[c][a0]);
            acc[0] = fmaf(x, m.x, acc[0]); acc[1] = fmaf(x, m.y, acc[1]);
            acc[2] = fmaf(x, m.z, acc[2]); acc[3] = fmaf(x, m.w, acc[3]);
        }
        *reinterpret_cast<float4 *>(&Un[i][a0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();
        *reinterpret_cast<float4 *>(&Ut[i][a0]) = *reinterpret_cast<const float4 *>(&Un[i][a0]);
        __syncthreads();
        const float4 u = emit(k);
        ub[0] = fmaf(p.w[k], u.x, ub[0]); ub[1] = fmaf(p.w[k], u.y, ub[1]);
        ub[2] = fmaf(p.w[k], u.z, ub[2]); ub[3] = fmaf(p.w[k], u.w, ub[3]);
    }
    // Ubar transposed and its bf16 hi + lo image (the tensor-core passes on this
    // path read no row-major fp32 copy); the adaptive weights' passes read none
    // of them (their walk terms are per token)
    if (b.mlp) return;
    *reinterpret_cast<float4 *>(b.UbarT + so + e * D + a0) = make_float4(ub[0], ub[1], ub[2], ub[3]);
    // the image is row-major (Ubar[a][e]): through shared memory, so that each row's
    // R entries of this CTA go out together
    *reinterpret_cast<float4 *>(&Un[i][a0]) = make_float4(ub[0], ub[1], ub[2], ub[3]);
    __syncthreads();
    for (int x = tid; x < D * R; x += kThreads) {
        const int a = x / R, ii = x % R;
        const float v = Un[ii][a];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        b.ubimg[so * 2 + a * D + e0 + ii] = __bfloat16_as_ushort(hi);
        b.ubimg[so * 2 + D * D + a * D + e0 + ii] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
    }
}

// ---------------------------------------------------------------------------
// 2. partial dUbar = sum_j Q~_j (alpha dO_j)^T over one chunk.
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_stats_dub(BwdProblem b) {
    constexpr int RB = D / 16;   // each thread: an RB x RB block of the D x D result
    __shared__ float Qs[kTile][D];
    __shared__ float Gs[kTile][D];
    __shared__ float s[D];
    const Problem &p = b.fwd;
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid < D) s[tid] = p.s_red[(size_t)sl * D + tid];
    __syncthreads();
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const TIn *Q = static_cast<const TIn *>(p.Q) + (size_t)sl * p.n * D;
    const TIn *dO = static_cast<const TIn *>(b.dO) + (size_t)sl * p.n * D;
    const float al = p.alpha[sl % p.heads];
    const int a0 = (tid / 16) * RB, e0 = (tid % 16) * RB;
    float acc[RB][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) acc[r][x] = 0.f;
    for (int base = t0; base < t1; base += kTile) {
        const int cnt = min(kTile, t1 - base);
        for (int idx = tid; idx < kTile * D; idx += kThreads) {
            const int j = idx / D, ch = idx % D;
            float qv = 0.f, gv = 0.f;
            if (j < cnt) {
                qv = feature(ld(Q + (size_t)(base + j) * D + ch), p.relu);
                gv = al * ld(dO + (size_t)(base + j) * D + ch);
            }
            Qs[j][ch] = qv;
            Gs[j][ch] = gv;
        }
        __syncthreads();
        for (int j = warp; j < kTile; j += kWarps) {   // Q~_j = Q_j / (Q_j . s + eps)
            float d = 0.f;
            for (int ch = lane; ch < D; ch += 32) d += Qs[j][ch] * s[ch];
            const float r = 1.f / (warp_sum(d) + p.eps);
            __syncwarp();
            for (int ch = lane; ch < D; ch += 32) Qs[j][ch] *= r;
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
            float ra[RB], rb[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                ra[r] = Qs[j][a0 + r];
                rb[r] = Gs[j][e0 + r];
            }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int x = 0; x < RB; ++x) acc[r][x] = fmaf(ra[r], rb[x], acc[r][x]);
        }
        __syncthreads();
    }
    float *out = b.dub_part + ((size_t)sl * p.chunks + c) * D * D;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) out[(a0 + r) * D + e0 + x] = acc[r][x];
}

// ---------------------------------------------------------------------------
// 2'. adaptive weights: partial dU_k = sum_j Q~_j (w_jk alpha dO_j)^T over one
// chunk, one k per blockIdx.y (k = 1 + blockIdx.y).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_stats_duk(BwdProblem b) {
    constexpr int RB = D / 16;
    __shared__ float Qs[kTile][D];
    __shared__ float Gs[kTile][D];
    __shared__ float s[D];
    const Problem &p = b.fwd;
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, k = 1 + blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid < D) s[tid] = p.s_red[(size_t)sl * D + tid];
    __syncthreads();
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const TIn *Q = static_cast<const TIn *>(p.Q) + (size_t)sl * p.n * D;
    const TIn *dO = static_cast<const TIn *>(b.dO) + (size_t)sl * p.n * D;
    const float *wt = b.wtok + (size_t)sl * p.n * p.T;
    const float al = p.alpha[sl % p.heads];
    const int a0 = (tid / 16) * RB, e0 = (tid % 16) * RB;
    float acc[RB][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) acc[r][x] = 0.f;
    for (int base = t0; base < t1; base += kTile) {
        const int cnt = min(kTile, t1 - base);
        for (int idx = tid; idx < kTile * D; idx += kThreads) {
            const int j = idx / D, ch = idx % D;
            float qv = 0.f, gv = 0.f;
            if (j < cnt) {
                qv = feature(ld(Q + (size_t)(base + j) * D + ch), p.relu);
                gv = al * wt[(size_t)(base + j) * p.T + k] * ld(dO + (size_t)(base + j) * D + ch);
            }
            Qs[j][ch] = qv;
            Gs[j][ch] = gv;
        }
        __syncthreads();
        for (int j = warp; j < kTile; j += kWarps) {   // Q~_j = Q_j / (Q_j . s + eps)
            float d = 0.f;
            for (int ch = lane; ch < D; ch += 32) d += Qs[j][ch] * s[ch];
            const float r = 1.f / (warp_sum(d) + p.eps);
            __syncwarp();
            for (int ch = lane; ch < D; ch += 32) Qs[j][ch] *= r;
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
            float ra[RB], rb[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                ra[r] = Qs[j][a0 + r];
                rb[r] = Gs[j][e0 + r];
            }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int x = 0; x < RB; ++x) acc[r][x] = fmaf(ra[r], rb[x], acc[r][x]);
        }
        __syncthreads();
    }
    float *out = b.dukp + (((size_t)sl * p.chunks + c) * b.nh + (k - 1)) * D * D;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) out[(a0 + r) * D + e0 + x] = acc[r][x];
}

// In-grid 3x3 window of token i on the H x W grid (the token itself first
// is not required; order is row-major over the offsets).
__device__ __forceinline__ int window(int i, int H, int W, int (&nb)[9]) {
    const int r = i / W, c = i % W;
    int cnt = 0;
    for (int dr = -1; dr <= 1; ++dr)
        for (int dc = -1; dc <= 1; ++dc) {
            const int rr = r + dr, cc = c + dc;
            if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue;
            nb[cnt++] = rr * W + cc;
        }
    return cnt;
}

// dL/dx from dL/dphi(x) through the feature map: ReLU passes x > 0 only,
// ELU(x) + 1 has slope exp(x) below 0.
__device__ __forceinline__ float feature_grad(float g, float x, int fmap) {
    if (fmap == 1) return x > 0.f ? g : 0.f;
    if (fmap == 2) return x > 0.f ? g : g * expf(x);
    return g;
}

// Warp sums of n independent per-lane partials, the butterflies interleaved so
// their shuffle latencies overlap.
template <int N>
__device__ __forceinline__ void warp_sum_n(float (&x)[N]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int t = 0; t < N; ++t) x[t] += __shfl_xor_sync(0xffffffffu, x[t], o);
}

// Lane l holds channels l and l + 32 (those below D).
template <typename TIn, int D>
__device__ __forceinline__ void load_row(const TIn *row, float (&x)[(D + 31) / 32], int lane, int relu) {
#pragma unroll
    for (int t = 0; t < (D + 31) / 32; ++t) {
        const int ch = lane + 32 * t;
        x[t] = ch < D ? feature(ld(row + ch), relu) : 0.f;
    }
}
template <int D>
__device__ __forceinline__ float dot_row(const float (&x)[(D + 31) / 32], const float (&y)[(D + 31) / 32]) {
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < (D + 31) / 32; ++t) acc = fmaf(x[t], y[t], acc);
    return warp_sum(acc);
}

// ---------------------------------------------------------------------------
// 3. per token: window softmax statistics (max, sum), dl_i . l_i, and the
// dalpha terms dO_i . (g_i - l_i), summed per block in a fixed order.
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_token_a(BwdProblem b) {
    constexpr int NC = (D + 31) / 32;
    __shared__ float part[kWarps];
    const Problem &p = b.fwd;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x / b.nblk, blk = blockIdx.x % b.nblk;
    const size_t sbase = (size_t)sl * p.n * D;
    const TIn *Q = static_cast<const TIn *>(p.Q) + sbase;
    const TIn *K = static_cast<const TIn *>(p.K) + sbase;
    const TIn *V = static_cast<const TIn *>(p.V) + sbase;
    const TIn *dO = static_cast<const TIn *>(b.dO) + sbase;
    const float *s = p.s_red + (size_t)sl * D;
    const float *Ub = b.Ubar + (size_t)sl * D * D;
    const float al = p.alpha[sl % p.heads], w0 = p.w[0];
    const float scale = rsqrtf((float)D);
    float dal = 0.f;
    for (int u = warp; u < b.tpb; u += kWarps) {
        const int i = blk * b.tpb + u;
        if (i >= p.n) break;
        float q[NC], v[NC], go[NC], sv[NC];
        load_row<TIn, D>(Q + (size_t)i * D, q, lane, p.relu);
        load_row<TIn, D>(V + (size_t)i * D, v, lane, 0);
        load_row<TIn, D>(dO + (size_t)i * D, go, lane, 0);
#pragma unroll
        for (int t = 0; t < NC; ++t) sv[t] = lane + 32 * t < D ? s[lane + 32 * t] : 0.f;
        const float rq = 1.f / (dot_row<D>(q, sv) + p.eps);
        // g_i = w_0 V_i + Q~_i Ubar
        float g[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) g[t] = 0.f;
        for (int a = 0; a < D; ++a) {
            const float qa = __shfl_sync(0xffffffffu, q[a / 32], a % 32);
#pragma unroll
            for (int t = 0; t < NC; ++t)
                if (lane + 32 * t < D) g[t] = fmaf(qa, Ub[(size_t)a * D + lane + 32 * t], g[t]);
        }
#pragma unroll
        for (int t = 0; t < NC; ++t) g[t] = fmaf(rq, g[t], w0 * v[t]);
        // local window: every neighbour row loaded, then the nine scores reduced together
        int nb[9];
        const int cnt = window(i, p.H, p.W, nb);
        float kr[9][NC], vr[9][NC], e[9];
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9) {
            const int row = t9 < cnt ? nb[t9] : i;
            load_row<TIn, D>(K + (size_t)row * D, kr[t9], lane, p.relu);
            load_row<TIn, D>(V + (size_t)row * D, vr[t9], lane, 0);
            e[t9] = 0.f;
#pragma unroll
            for (int t = 0; t < NC; ++t) e[t9] = fmaf(q[t], kr[t9][t], e[t9]);
        }
        warp_sum_n(e);
        float emax = -INFINITY;
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9)
            if (t9 < cnt) emax = fmaxf(emax, e[t9] * scale);
        float l[NC], esum = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) l[t] = 0.f;
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9) {
            if (t9 >= cnt) break;
            const float a = expf(e[t9] * scale - emax);
            esum += a;
#pragma unroll
            for (int t = 0; t < NC; ++t) l[t] = fmaf(a, vr[t9][t], l[t]);
        }
        const float inv = 1.f / esum;
        float dgl = 0.f, dll = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            l[t] *= inv;
            dgl = fmaf(go[t], g[t] - l[t], dgl);
            dll = fmaf(go[t], l[t], dll);
        }
        float red[2] = {dgl, dll};
        warp_sum_n(red);
        dgl = red[0];
        dll = red[1] * (1.f - al);
        dal += dgl;
        if (lane == 0)
            reinterpret_cast<float4 *>(b.lstat)[(size_t)sl * p.n + i] = make_float4(emax, esum, dll, 0.f);
    }
    if (lane == 0) part[warp] = dal;
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int w = 0; w < kWarps; ++w) acc += part[w];
        b.dal_part[(size_t)sl * b.nblk + blk] = acc;
    }
}

// ---------------------------------------------------------------------------
// 3'. adaptive weights, per token i (replaces bwd_token_a): the window's
// softmax statistics and the dalpha terms as there, with the token's own
// weights; and the MLP's backward:
//   x_i = [q_i; k_i], a_i = W1 x_i + b1, h_i = GELU(a_i), w_i = softmax(W2 h_i + b2)
//   dw_ik = alpha dO_i . Y_k,i (Y_0 = V_i, Y_k = Q~_i U_k), dz_i = w_i (dw_i - w_i . dw_i)
//   da_i = (W2^T dz_i) GELU'(a_i),  the MLP's share of [dq_i; dk_i] = W1^T da_i
// Stored per token: w_i and dz_i (T), h_i and da_i (hidden), the share (2 d).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float gelu_exact(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_exact_grad(float x) {
    return 0.5f * (1.f + erff(x * 0.70710678118654752f)) + x * 0.39894228040143268f * expf(-0.5f * x * x);
}

template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_token_mlp(BwdProblem b) {
    constexpr int NC = (D + 31) / 32;
    constexpr int TM = LISA_MAX_T_MLP;
    __shared__ float part[kWarps];
    __shared__ float pre_s[kWarps][LISA_MAX_HIDDEN];
    __shared__ float h_s[kWarps][LISA_MAX_HIDDEN];
    __shared__ float da_s[kWarps][LISA_MAX_HIDDEN];
    const Problem &p = b.fwd;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x / b.nblk, blk = blockIdx.x % b.nblk;
    const int T = p.T, hid = p.hidden;
    const size_t sbase = (size_t)sl * p.n * D;
    const TIn *Q = static_cast<const TIn *>(p.Q) + sbase;
    const TIn *K = static_cast<const TIn *>(p.K) + sbase;
    const TIn *V = static_cast<const TIn *>(p.V) + sbase;
    const TIn *dO = static_cast<const TIn *>(b.dO) + sbase;
    const float *s = p.s_red + (size_t)sl * D;
    const float al = p.alpha[sl % p.heads];
    const float scale = rsqrtf((float)D);
    float dal = 0.f;
    for (int u = warp; u < b.tpb; u += kWarps) {
        const int i = blk * b.tpb + u;
        if (i >= p.n) break;
        float q[NC], k[NC], v[NC], go[NC], sv[NC];
        load_row<TIn, D>(Q + (size_t)i * D, q, lane, p.relu);
        load_row<TIn, D>(K + (size_t)i * D, k, lane, p.relu);
        load_row<TIn, D>(V + (size_t)i * D, v, lane, 0);
        load_row<TIn, D>(dO + (size_t)i * D, go, lane, 0);
#pragma unroll
        for (int t = 0; t < NC; ++t) sv[t] = lane + 32 * t < D ? s[lane + 32 * t] : 0.f;
        const float rq = 1.f / (dot_row<D>(q, sv) + p.eps);
        // the MLP forward (pre-activations and h in shared memory, per warp)
        for (int m = 0; m < hid; ++m) {
            const float *row = p.W1 + (size_t)m * 2 * D;
            float acc = 0.f;
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                const int ch = lane + 32 * t;
                if (ch < D) acc = fmaf(row[ch], q[t], fmaf(row[D + ch], k[t], acc));
            }
            acc = warp_sum(acc) + p.b1[m];
            if (lane == 0) {
                pre_s[warp][m] = acc;
                h_s[warp][m] = gelu_exact(acc);
            }
        }
        __syncwarp();
        float w[TM], zmax = -INFINITY, zs = 0.f;
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            w[t] = 0.f;
            if (t < T) {
                float z = p.b2[t];
                for (int m = 0; m < hid; ++m) z = fmaf(p.W2[(size_t)t * hid + m], h_s[warp][m], z);
                w[t] = z;
                zmax = fmaxf(zmax, z);
            }
        }
#pragma unroll
        for (int t = 0; t < TM; ++t)
            if (t < T) {
                w[t] = expf(w[t] - zmax);
                zs += w[t];
            }
        const float izs = 1.f / zs;
#pragma unroll
        for (int t = 0; t < TM; ++t) w[t] = t < T ? w[t] * izs : 0.f;
        // walk terms Y_k (k >= 1), g_i, and the partial sums of dw
        float g[NC], dw[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) dw[t] = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            g[t] = w[0] * v[t];
            dw[0] = fmaf(al * go[t], v[t], dw[0]);
        }
#pragma unroll
        for (int kk = 1; kk < TM; ++kk) {
            if (kk >= T) break;
            const float *Un = b.Ukn + ((size_t)sl * b.nh + (kk - 1)) * D * D;
            float y[NC];
#pragma unroll
            for (int t = 0; t < NC; ++t) y[t] = 0.f;
            for (int a = 0; a < D; ++a) {
                const float qa = __shfl_sync(0xffffffffu, q[a / 32], a % 32) * rq;
#pragma unroll
                for (int t = 0; t < NC; ++t)
                    if (lane + 32 * t < D) y[t] = fmaf(qa, Un[(size_t)a * D + lane + 32 * t], y[t]);
            }
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                g[t] = fmaf(w[kk], y[t], g[t]);
                dw[kk] = fmaf(al * go[t], y[t], dw[kk]);
            }
        }
        warp_sum_n(dw);
        // local window (as bwd_token_a)
        int nb[9];
        const int cnt = window(i, p.H, p.W, nb);
        float kr[9][NC], vr[9][NC], e[9];
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9) {
            const int row = t9 < cnt ? nb[t9] : i;
            load_row<TIn, D>(K + (size_t)row * D, kr[t9], lane, p.relu);
            load_row<TIn, D>(V + (size_t)row * D, vr[t9], lane, 0);
            e[t9] = 0.f;
#pragma unroll
            for (int t = 0; t < NC; ++t) e[t9] = fmaf(q[t], kr[t9][t], e[t9]);
        }
        warp_sum_n(e);
        float emax = -INFINITY;
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9)
            if (t9 < cnt) emax = fmaxf(emax, e[t9] * scale);
        float l[NC], esum = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) l[t] = 0.f;
#pragma unroll
        for (int t9 = 0; t9 < 9; ++t9) {
            if (t9 >= cnt) break;
            const float a = expf(e[t9] * scale - emax);
            esum += a;
#pragma unroll
            for (int t = 0; t < NC; ++t) l[t] = fmaf(a, vr[t9][t], l[t]);
        }
        const float inv = 1.f / esum;
        float red[2] = {0.f, 0.f};
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            l[t] *= inv;
            red[0] = fmaf(go[t], g[t] - l[t], red[0]);
            red[1] = fmaf(go[t], l[t], red[1]);
        }
        warp_sum_n(red);
        dal += red[0];
        const size_t ti = (size_t)sl * p.n + i;
        if (lane == 0) reinterpret_cast<float4 *>(b.lstat)[ti] = make_float4(emax, esum, red[1] * (1.f - al), 0.f);
        // softmax and MLP backward
        float wdw = 0.f, dz[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) wdw = fmaf(w[t], dw[t], wdw);
#pragma unroll
        for (int t = 0; t < TM; ++t) dz[t] = w[t] * (dw[t] - wdw);
        for (int m = lane; m < hid; m += 32) {
            float dh = 0.f;
#pragma unroll
            for (int t = 0; t < TM; ++t)
                if (t < T) dh = fmaf(p.W2[(size_t)t * hid + m], dz[t], dh);
            da_s[warp][m] = dh * gelu_exact_grad(pre_s[warp][m]);
            b.hbuf[ti * hid + m] = h_s[warp][m];
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < TM; ++t)
            if (t < T && lane == t) {
                b.wtok[ti * T + t] = w[t];
                b.dzbuf[ti * T + t] = dz[t];
            }
        for (int m = lane; m < hid; m += 32) b.dabuf[ti * hid + m] = da_s[warp][m];
        for (int c = lane; c < 2 * D; c += 32) {
            float acc = 0.f;
            for (int m = 0; m < hid; ++m) acc = fmaf(p.W1[(size_t)m * 2 * D + c], da_s[warp][m], acc);
            b.dxm[ti * 2 * D + c] = acc;
        }
        __syncwarp();   // the next token of this warp rewrites pre_s, h_s, da_s
    }
    if (lane == 0) part[warp] = dal;
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int w2 = 0; w2 < kWarps; ++w2) acc += part[w2];
        b.dal_part[(size_t)sl * b.nblk + blk] = acc;
    }
}

// ---------------------------------------------------------------------------
// 4. reduce dUbar; the walk's backward recurrence (or the transposed solve)
// gives dM and dU_1.
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// 4 (d = 64, truncated walk). The reverse recurrence of step 4 with every
// 64 x 64 product register-blocked in shared memory (U_(k-1) staged, not
// read from global memory in the inner loop).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) bwd_recur_back_64(BwdProblem b) {
    constexpr int D = 64;
    __shared__ __align__(16) float M[D * D];
    __shared__ __align__(16) float G[D * D];
    __shared__ __align__(16) float X[D * D];
    const Problem &p = b.fwd;
    const int sl = blockIdx.x, tid = threadIdx.x;
    const int a0 = 4 * (tid >> 4), c0 = 4 * (tid & 15);
    const size_t so = (size_t)sl * D * D;
    // reduced dUbar at the thread's block (chunk order), M staged
    float dub[4][4];
    const int parts = b.tc_dub ? b.tcfwd.chunks / b.tcfwd.tc_cluster : 0;
    const float al = p.alpha[sl % p.heads];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b.tc_dub) {   // alpha (Q~^T dO): rows 64 + a of the tensor-core partials, in part order
            for (int q = 0; q < parts; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(
                    b.tcdub + ((size_t)sl * parts + q) * 2 * D * D + (D + a0 + i) * D + c0);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            acc.x *= al; acc.y *= al; acc.z *= al; acc.w *= al;
        } else if (!b.mlp) {
            for (int c = 0; c < p.chunks; ++c) {
                const float4 v = *reinterpret_cast<const float4 *>(
                    b.dub_part + ((size_t)sl * p.chunks + c) * D * D + (a0 + i) * D + c0);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
        }
        dub[i][0] = acc.x; dub[i][1] = acc.y; dub[i][2] = acc.z; dub[i][3] = acc.w;
    }
    for (int x = tid; x < D * D / 4; x += kThreads)
        reinterpret_cast<float4 *>(M)[x] = reinterpret_cast<const float4 *>(b.Mred + so)[x];
    // the direct term of dL/dU_k on the thread's block: w_k dUbar, or with the
    // adaptive weights sum_i w_ik Q~_i^T dg_i (its split-K partials, in chunk order)
    auto level = [&](int k, float (&out)[4][4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) out[i][j] = b.mlp ? 0.f : p.w[k] * dub[i][j];
        if (b.mlp)
            for (int c = 0; c < p.chunks; ++c)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        b.dukp + (((size_t)sl * p.chunks + c) * b.nh + (k - 1)) * D * D + (a0 + i) * D + c0);
                    out[i][0] += v.x; out[i][1] += v.y; out[i][2] += v.z; out[i][3] += v.w;
                }
    };
    const float *Uk = b.Uk + (size_t)sl * b.nh * D * D;   // transposed: Uk[e][c] = U_k[c][e]
    float dm[4][4], g[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) dm[i][j] = g[i][j] = 0.f;
    if (p.T > 1) {
        level(p.T - 1, g);
#pragma unroll
        for (int i = 0; i < 4; ++i) st_row4(G + (a0 + i) * D + c0, g[i]);
        for (int k = p.T - 1; k >= 2; --k) {
            // dM += G_k U_(k-1)^T: B(e, c) = U_(k-1)[c][e], staged from the transposed copy
            const float4 *Up = reinterpret_cast<const float4 *>(Uk + (size_t)(k - 2) * D * D);
            for (int x = tid; x < D * D / 4; x += kThreads) reinterpret_cast<float4 *>(X)[x] = Up[x];
            __syncthreads();
            mm64_acc<false>(G, X, dm, tid);
            // G_(k-1) = (direct term of U_(k-1)) + M^T G_k
            level(k - 1, g);
            mm64_acc<true>(M, G, g, tid);
            __syncthreads();   // every read of G and X done
#pragma unroll
            for (int i = 0; i < 4; ++i) st_row4(G + (a0 + i) * D + c0, g[i]);
        }
        __syncthreads();
    }
    // outputs: dM, dU_1 = G_1 and their transposes
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        st_row4(b.dM + so + (a0 + i) * D + c0, dm[i]);
        st_row4(b.dU1 + so + (a0 + i) * D + c0, g[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            b.dMT[so + (c0 + j) * D + a0 + i] = dm[i][j];
            b.dU1T[so + (c0 + j) * D + a0 + i] = g[i][j];
        }
    }
}

// ---------------------------------------------------------------------------
// 4'' (d = 64, truncated walk, T <= 3, fixed weights, dUbar from the
// tensor-core partials): the reverse recurrence split over kRecurSplit CTAs
// per slice.  With T <= 3 there is at most one step: G_2 = w_2 dUbar,
// dM = G_2 U_1^T and dU_1 = G_1 = w_1 dUbar + M^T G_2, so rows e0 .. e0 + 15
// of dM and dU_1 need only the whole dUbar, M and U_1.  Each CTA reduces the
// whole dUbar (in the same order as bwd_recur_back_64, so the bits agree) and
// computes its own rows.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) bwd_recur_back_rows(BwdProblem b) {
    constexpr int D = 64, R = D / kRecurSplit;
    __shared__ __align__(16) float M[D * D];   // M row-major: M[e * D + a] = M[e][a]
    __shared__ __align__(16) float G[D * D];   // dUbar, row-major
    __shared__ __align__(16) float X[D * D];   // U_1 transposed: X[e * D + c] = U_1[c][e]
    const Problem &p = b.fwd;
    const int sl = blockIdx.x / kRecurSplit, e0 = R * (blockIdx.x % kRecurSplit), tid = threadIdx.x;
    const size_t so = (size_t)sl * D * D;
    const int parts = b.tcfwd.chunks / b.tcfwd.tc_cluster;
    const float al = p.alpha[sl % p.heads];
    for (int x = tid; x < D * D / 4; x += kThreads) {   // alpha (Q~^T dO): rows 64 + a of the partials
        const int a = x / 16, c4 = (x % 16) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < parts; ++q) {
            const float4 v =
                *reinterpret_cast<const float4 *>(b.tcdub + ((size_t)sl * parts + q) * 2 * D * D + (D + a) * D + c4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        acc.x *= al; acc.y *= al; acc.z *= al; acc.w *= al;
        *reinterpret_cast<float4 *>(G + a * D + c4) = acc;
        reinterpret_cast<float4 *>(M)[x] = reinterpret_cast<const float4 *>(b.Mred + so)[x];
        if (p.T > 2)   // U_1 (k = 1 of the transposed copies)
            reinterpret_cast<float4 *>(X)[x] = reinterpret_cast<const float4 *>(b.Uk + (size_t)sl * b.nh * D * D)[x];
    }
    __syncthreads();
    // thread: row a = e0 + tid / 16, columns c0 .. c0 + 3
    const int a = e0 + (tid >> 4), c0 = 4 * (tid & 15);
    const float w1 = p.T > 1 ? p.w[1] : 0.f, w2 = p.T > 2 ? p.w[2] : 0.f;
    float g[4], dm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = w1 * G[a * D + c0 + j];
    if (p.T > 2) {
#pragma unroll 4
        for (int e = 0; e < D; ++e) {
            const float ga = w2 * G[a * D + e];   // G_2[a][e]
            const float me = M[e * D + a];        // M[e][a]
            const float4 xv = *reinterpret_cast<const float4 *>(X + e * D + c0);
            const float4 gv = *reinterpret_cast<const float4 *>(G + e * D + c0);
            dm[0] = fmaf(ga, xv.x, dm[0]); dm[1] = fmaf(ga, xv.y, dm[1]);
            dm[2] = fmaf(ga, xv.z, dm[2]); dm[3] = fmaf(ga, xv.w, dm[3]);
            g[0] = fmaf(me, w2 * gv.x, g[0]); g[1] = fmaf(me, w2 * gv.y, g[1]);
            g[2] = fmaf(me, w2 * gv.z, g[2]); g[3] = fmaf(me, w2 * gv.w, g[3]);
        }
    }
    st_row4(b.dM + so + a * D + c0, dm);
    st_row4(b.dU1 + so + a * D + c0, g);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        b.dMT[so + (c0 + j) * D + a] = dm[j];
        b.dU1T[so + (c0 + j) * D + a] = g[j];
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_recur_back(BwdProblem b) {
    constexpr int EPT = D * D / kThreads;
    __shared__ float M[D][D];
    __shared__ float G[D][D];
    __shared__ float X[D][D];
    const Problem &p = b.fwd;
    const int sl = blockIdx.x, tid = threadIdx.x;
    float dub[EPT];
#pragma unroll
    for (int x = 0; x < EPT; ++x) {
        const int idx = tid + x * kThreads;
        float acc = 0.f;
        if (!b.mlp)
            for (int c = 0; c < p.chunks; ++c) acc += b.dub_part[((size_t)sl * p.chunks + c) * D * D + idx];
        dub[x] = acc;
        M[idx / D][idx % D] = b.Mred[(size_t)sl * D * D + idx];
    }
    // the direct term of dL/dU_k at entry x: w_k dUbar, or with the adaptive
    // weights sum_i w_ik Q~_i^T dg_i (its split-K partials, in chunk order)
    auto level = [&](int k, int x) -> float {
        if (!b.mlp) return p.w[k] * dub[x];
        const int idx = tid + x * kThreads;
        float acc = 0.f;
        for (int c = 0; c < p.chunks; ++c)
            acc += b.dukp[(((size_t)sl * p.chunks + c) * b.nh + (k - 1)) * D * D + idx];
        return acc;
    };
    float *dM = b.dM + (size_t)sl * D * D, *dU1 = b.dU1 + (size_t)sl * D * D;
    const float *Uk = b.Uk + (size_t)sl * b.nh * D * D;   // transposed
    __syncthreads();
    if (p.untruncated) {
        // (I - beta M)^T Y = beta (1-beta) dUbar: A' = (I - beta M)^T by
        // columns is I - beta M by rows (in G); R = the right side by columns (in X)
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int a = idx / D, c = idx % D;
            G[a][c] = (a == c ? 1.f : 0.f) - p.beta * M[a][c];
        }
#pragma unroll
        for (int x = 0; x < EPT; ++x) {
            const int idx = tid + x * kThreads;
            X[idx % D][idx / D] = p.beta * (1.f - p.beta) * dub[x];
        }
        __syncthreads();
        solve_walk_system<kWarps, (2 * D + kWarps - 1) / kWarps>(&G[0][0], D, &X[0][0], D, D, D, &M[0][0], tid);
        // dU_1 = Y; dM = beta Y Z^T with Z = U_1's slot (the solved Z)
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int a = idx / D, c = idx % D;
            dU1[idx] = X[c][a];
            float acc = 0.f;
            for (int e = 0; e < D; ++e) acc = fmaf(X[e][a], Uk[(size_t)e * D + c], acc);
            dM[idx] = p.beta * acc;
            b.dMT[(size_t)sl * D * D + c * D + a] = p.beta * acc;
            b.dU1T[(size_t)sl * D * D + c * D + a] = X[c][a];
        }
        return;
    }
    float dm[EPT];
#pragma unroll
    for (int x = 0; x < EPT; ++x) dm[x] = 0.f;
    if (p.T > 1) {
#pragma unroll
        for (int x = 0; x < EPT; ++x) {
            const int idx = tid + x * kThreads;
            G[idx / D][idx % D] = level(p.T - 1, x);
        }
        __syncthreads();
        for (int k = p.T - 1; k >= 2; --k) {
            // dM += G_k U_(k-1)^T, then G_(k-1) = (direct term of U_(k-1)) + M^T G_k
            const float *Up = Uk + (size_t)(k - 2) * D * D;
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const int a = idx / D, c = idx % D;
                float acc = 0.f;
                for (int e = 0; e < D; ++e) acc = fmaf(G[a][e], Up[(size_t)e * D + c], acc);
                dm[x] += acc;
            }
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const int a = idx / D, e = idx % D;
                float acc = level(k - 1, x);
                for (int c = 0; c < D; ++c) acc = fmaf(M[c][a], G[c][e], acc);
                X[a][e] = acc;
            }
            __syncthreads();
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                G[idx / D][idx % D] = X[idx / D][idx % D];
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int x = 0; x < EPT; ++x) {
        const int idx = tid + x * kThreads;
        const int a = idx / D, c = idx % D;
        const float u1 = p.T > 1 ? G[a][c] : 0.f;
        dM[idx] = dm[x];
        dU1[idx] = u1;
        b.dMT[(size_t)sl * D * D + c * D + a] = dm[x];
        b.dU1T[(size_t)sl * D * D + c * D + a] = u1;
    }
}

// ---------------------------------------------------------------------------
// 5. per token j: dXq_j, dV_j, the ds terms -c_j Q_j (per-block sums), and
// dK_j without ds (fp32).  The block's kTpb tokens first go through the three
// d x d products together, from shared memory:
//   dQ~_j = alpha dO_j Ubar^T + K_j dM,  dV_j = w_0 alpha dO_j + K_j dU_1,
//   dK_j  = V_j dU_1^T + Q~_j dM^T
// (thread: 4 channels x the tokens of its group), then one warp per token
// takes the normaliser, the window and the stores.
// ---------------------------------------------------------------------------
// Adaptive weights: the token's own walk terms, which the block's shared
// products leave out (they see w = 0 and Ubar = 0):
//   dV_j += w_j0 alpha dO_j,  dQ~_j += alpha sum_{k>=1} w_jk dO_j U_k^T
// U_k^T is read from the transposed copy (coalesced over the output channel).
template <int D>
__device__ __forceinline__ void mlp_walk_terms(const BwdProblem &b, int sl, int j, int lane, float al,
                                               const float (&go)[(D + 31) / 32], float (&dqt)[(D + 31) / 32],
                                               float (&dv)[(D + 31) / 32]) {
    constexpr int NC = (D + 31) / 32;
    const int T = b.fwd.T;
    const float *wt = b.wtok + ((size_t)sl * b.fwd.n + j) * T;
#pragma unroll
    for (int t = 0; t < NC; ++t) dv[t] = fmaf(wt[0] * al, go[t], dv[t]);
    for (int kk = 1; kk < T; ++kk) {
        const float wk = al * wt[kk];
        const float *UT = b.Uk + ((size_t)sl * b.nh + (kk - 1)) * D * D;   // UT[c][a] = U_k[a][c]
        for (int c = 0; c < D; ++c) {
            const float gc = __shfl_sync(0xffffffffu, go[c / 32], c % 32) * wk;
#pragma unroll
            for (int t = 0; t < NC; ++t)
                if (lane + 32 * t < D) dqt[t] = fmaf(gc, UT[(size_t)c * D + lane + 32 * t], dqt[t]);
        }
    }
}

constexpr int kTpb = 32;   // tokens per block of the per-token kernels

template <int D>
constexpr int token_b_smem_floats() { return 5 * D * D + 7 * kTpb * D; }

template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_token_b(BwdProblem b) {
    constexpr int NC = (D + 31) / 32;
    constexpr int CG = D / 4;                    // channel groups of 4
    constexpr int TG = kThreads / CG;            // token groups
    extern __shared__ float4 smem_b[];
    float *UbT = reinterpret_cast<float *>(smem_b);
    float *dMs = UbT + D * D, *dU1s = dMs + D * D, *dU1T = dU1s + D * D, *dMT = dU1T + D * D;
    float *Qr = dMT + D * D, *Gr = Qr + kTpb * D, *Kr = Gr + kTpb * D, *Vr = Kr + kTpb * D;
    float *oQ = Vr + kTpb * D, *oV = oQ + kTpb * D, *oK = oV + kTpb * D;
    __shared__ float rqs[kTpb];
    __shared__ float dsw[kWarps][D];
    const Problem &p = b.fwd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = blockIdx.x / b.nblk, blk = blockIdx.x % b.nblk;
    const int j0 = blk * kTpb, cnt = min(kTpb, p.n - j0);
    const size_t sbase = (size_t)sl * p.n * D;
    const TIn *Q = static_cast<const TIn *>(p.Q) + sbase;
    const TIn *K = static_cast<const TIn *>(p.K) + sbase;
    const TIn *V = static_cast<const TIn *>(p.V) + sbase;
    const TIn *dO = static_cast<const TIn *>(b.dO) + sbase;
    TIn *dQo = static_cast<TIn *>(b.dQ) + sbase;
    TIn *dVo = static_cast<TIn *>(b.dV) + sbase;
    float *dKp = b.dk_part + sbase;
    const float4 *lst = reinterpret_cast<const float4 *>(b.lstat) + (size_t)sl * p.n;
    const float *s = p.s_red + (size_t)sl * D;
    const float al = p.alpha[sl % p.heads], w0 = p.w[0];
    const float scale = rsqrtf((float)D);

    // ---- stage the slice's matrices and the block's token rows
    {
        const size_t mo = (size_t)sl * D * D / 4;
        const float4 *src[5] = {reinterpret_cast<const float4 *>(b.UbarT) + mo,
                                reinterpret_cast<const float4 *>(b.dM) + mo,
                                reinterpret_cast<const float4 *>(b.dU1) + mo,
                                reinterpret_cast<const float4 *>(b.dU1T) + mo,
                                reinterpret_cast<const float4 *>(b.dMT) + mo};
#pragma unroll
        for (int m = 0; m < 5; ++m)
            for (int x = tid; x < D * D / 4; x += kThreads) smem_b[m * D * D / 4 + x] = src[m][x];
    }
    for (int x = tid; x < kTpb * D; x += kThreads) {
        const int j = x / D, ch = x % D;
        float q = 0.f, g = 0.f, k = 0.f, v = 0.f;
        if (j < cnt) {
            const size_t o = (size_t)(j0 + j) * D + ch;
            q = feature(ld(Q + o), p.relu);
            g = ld(dO + o);
            k = feature(ld(K + o), p.relu);
            v = ld(V + o);
        }
        Qr[x] = q;
        Gr[x] = g;
        Kr[x] = k;
        Vr[x] = v;
    }
    __syncthreads();
    for (int j = warp; j < kTpb; j += kWarps) {   // 1 / (Q_j . s + eps)
        float d = 0.f;
        for (int ch = lane; ch < D; ch += 32) d += Qr[j * D + ch] * s[ch];
        d = warp_sum(d);
        if (lane == 0) rqs[j] = 1.f / (d + p.eps);
    }
    __syncthreads();

    // ---- the three products: thread = channels 4 cg .. 4 cg + 3 of tokens tg, tg + TG, ...
    {
        const int cg = tid % CG, tg = tid / CG;
        for (int j = tg; j < kTpb; j += TG) {
            float4 dq = make_float4(0.f, 0.f, 0.f, 0.f), dv = dq, dk = dq;
            const float rq = rqs[j];
            for (int c = 0; c < D; ++c) {
                const float go = al * Gr[j * D + c], kc = Kr[j * D + c], vc = Vr[j * D + c];
                const float qc = Qr[j * D + c] * rq;
                const float4 ub = reinterpret_cast<const float4 *>(UbT + c * D)[cg];
                const float4 dm = reinterpret_cast<const float4 *>(dMs + c * D)[cg];
                const float4 du = reinterpret_cast<const float4 *>(dU1s + c * D)[cg];
                const float4 duT = reinterpret_cast<const float4 *>(dU1T + c * D)[cg];
                const float4 dmT = reinterpret_cast<const float4 *>(dMT + c * D)[cg];
                dq.x = fmaf(go, ub.x, fmaf(kc, dm.x, dq.x));
                dq.y = fmaf(go, ub.y, fmaf(kc, dm.y, dq.y));
                dq.z = fmaf(go, ub.z, fmaf(kc, dm.z, dq.z));
                dq.w = fmaf(go, ub.w, fmaf(kc, dm.w, dq.w));
                dv.x = fmaf(kc, du.x, dv.x);
                dv.y = fmaf(kc, du.y, dv.y);
                dv.z = fmaf(kc, du.z, dv.z);
                dv.w = fmaf(kc, du.w, dv.w);
                dk.x = fmaf(vc, duT.x, fmaf(qc, dmT.x, dk.x));
                dk.y = fmaf(vc, duT.y, fmaf(qc, dmT.y, dk.y));
                dk.z = fmaf(vc, duT.z, fmaf(qc, dmT.z, dk.z));
                dk.w = fmaf(vc, duT.w, fmaf(qc, dmT.w, dk.w));
            }
            reinterpret_cast<float4 *>(oQ + j * D)[cg] = dq;
            reinterpret_cast<float4 *>(oV + j * D)[cg] = dv;
            reinterpret_cast<float4 *>(oK + j * D)[cg] = dk;
        }
    }
    __syncthreads();

    // ---- one warp per token: normaliser, window, stores
    float ds[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) ds[t] = 0.f;
    for (int u = warp; u < cnt; u += kWarps) {
        const int j = j0 + u;
        float q[NC], k[NC], v[NC], go[NC], sv[NC], dqt[NC], dv[NC], dk[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            const int ch = lane + 32 * t;
            const bool in = ch < D;
            q[t] = in ? Qr[u * D + ch] : 0.f;
            k[t] = in ? Kr[u * D + ch] : 0.f;
            v[t] = in ? Vr[u * D + ch] : 0.f;
            go[t] = in ? Gr[u * D + ch] : 0.f;
            sv[t] = in ? s[ch] : 0.f;
            dqt[t] = in ? oQ[u * D + ch] : 0.f;
            dv[t] = in ? fmaf(w0 * al, go[t], oV[u * D + ch]) : 0.f;
            dk[t] = in ? oK[u * D + ch] : 0.f;
        }
        if (b.mlp) mlp_walk_terms<D>(b, sl, j, lane, al, go, dqt, dv);
        const float rq = rqs[u];
        // through Q~ = Q / r:  c_j = (dQ~_j . Q_j) / r_j^2
        const float cj = dot_row<D>(dqt, q) * rq * rq;
        float dq[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            dq[t] = dqt[t] * rq - cj * sv[t];
            ds[t] = fmaf(-cj, q[t], ds[t]);
        }
        if (b.mlp) {   // the MLP's share of dq_j, dk_j
            const float *xm = b.dxm + ((size_t)sl * p.n + j) * 2 * D;
#pragma unroll
            for (int t = 0; t < NC; ++t)
                if (lane + 32 * t < D) {
                    dq[t] += xm[lane + 32 * t];
                    dk[t] += xm[D + lane + 32 * t];
                }
        }
        // local window: j as the query (its own softmax row) and as a key /
        // value of each neighbour i's row (N is symmetric).  All neighbour
        // rows are loaded first; the 36 dot products are reduced together.
        int nb[9];
        const int nn = window(j, p.H, p.W, nb);
        const float4 sj = lst[j];
        const float izj = 1.f / sj.y;
        {
            float kr[9][NC], vr[9][NC], d1[18];
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                const int row = t9 < nn ? nb[t9] : j;
                load_row<TIn, D>(K + (size_t)row * D, kr[t9], lane, p.relu);
                load_row<TIn, D>(V + (size_t)row * D, vr[t9], lane, 0);
                d1[t9] = d1[9 + t9] = 0.f;
#pragma unroll
                for (int t = 0; t < NC; ++t) {
                    d1[t9] = fmaf(q[t], kr[t9][t], d1[t9]);
                    d1[9 + t9] = fmaf(go[t], vr[t9][t], d1[9 + t9]);
                }
            }
            warp_sum_n(d1);
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                if (t9 >= nn) break;
                const float a = expf(d1[t9] * scale - sj.x) * izj;
                const float de = a * (d1[9 + t9] * (1.f - al) - sj.z) * scale;
#pragma unroll
                for (int t = 0; t < NC; ++t) dq[t] = fmaf(de, kr[t9][t], dq[t]);
            }
        }
        {
            float qi[9][NC], gi[9][NC], d2[18];
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                const int row = t9 < nn ? nb[t9] : j;
                load_row<TIn, D>(Q + (size_t)row * D, qi[t9], lane, p.relu);
                load_row<TIn, D>(dO + (size_t)row * D, gi[t9], lane, 0);
                d2[t9] = d2[9 + t9] = 0.f;
#pragma unroll
                for (int t = 0; t < NC; ++t) {
                    d2[t9] = fmaf(qi[t9][t], k[t], d2[t9]);
                    d2[9 + t9] = fmaf(gi[t9][t], v[t], d2[9 + t9]);
                }
            }
            warp_sum_n(d2);
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                if (t9 >= nn) break;
                const float4 si = lst[nb[t9]];
                const float a = expf(d2[t9] * scale - si.x) / si.y;
                const float de = a * (d2[9 + t9] * (1.f - al) - si.z) * scale;
#pragma unroll
                for (int t = 0; t < NC; ++t) {
                    dv[t] = fmaf(a * (1.f - al), gi[t9][t], dv[t]);
                    dk[t] = fmaf(de, qi[t9][t], dk[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            const int ch = lane + 32 * t;
            if (ch < D) {
                const float xq = ld(Q + (size_t)j * D + ch);
                st(dQo + (size_t)j * D + ch, feature_grad(dq[t], xq, p.relu));
                st(dVo + (size_t)j * D + ch, dv[t]);
                dKp[(size_t)j * D + ch] = dk[t];
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NC; ++t)
        if (lane + 32 * t < D) dsw[warp][lane + 32 * t] = ds[t];
    __syncthreads();
    for (int ch = tid; ch < D; ch += kThreads) {
        float acc = 0.f;
        for (int w = 0; w < kWarps; ++w) acc += dsw[w][ch];
        b.ds_part[((size_t)sl * b.nblk + blk) * D + ch] = acc;
    }
}

// ---------------------------------------------------------------------------
// 5'. bf16, d = 64: the B operands of the tiled token pass's three d x d
// products (mma.sync m16n8k16, bf16 operands, fp32 accumulation)
//   dQ~ = [dO | K] [alpha Ubar^T ; dM],  dK = [V | Q~] [dU_1^T ; dM^T],  dV = K dU_1
// as one bf16 image per slice, built once per backward (bwd_bimg); Q~ is
// rounded to bf16 as an operand, the inputs are bf16 already.
// ---------------------------------------------------------------------------
constexpr int kImgRows = 5 * 64;   // [alpha Ubar^T; dM; dU_1^T; dM^T; dU_1], 64 columns each
constexpr int kBS = 72;            // B-image row stride in shared memory, bf16 (144 B: ldmatrix conflict-free)

// grid (slices, 5): block (sl, m) converts matrix m of slice sl, four floats per thread and step
__global__ void __launch_bounds__(kThreads) bwd_bimg(BwdProblem b) {
    const int sl = blockIdx.x, m = blockIdx.y;
    const size_t mo = (size_t)sl * 64 * 64;
    // adaptive weights: alpha U_1^T stands where alpha Ubar^T does (the tiled pass
    // scales that half of its first product by each token's w_1)
    const float *srcs[5] = {b.mlp ? b.Uk + (size_t)sl * b.nh * 64 * 64 : b.UbarT + mo, b.dM + mo, b.dU1T + mo,
                            b.dMT + mo, b.dU1 + mo};
    const float4 *src = reinterpret_cast<const float4 *>(srcs[m]);
    const float f = m == 0 ? b.fwd.alpha[sl % b.fwd.heads] : 1.f;
    uint2 *img = reinterpret_cast<uint2 *>(b.bimg + ((size_t)sl * kImgRows + (size_t)m * 64) * 64);
    for (int x = threadIdx.x; x < 64 * 64 / 4; x += kThreads) {
        const float4 v = src[x];
        img[x] = make_uint2(sm100::pack_bf16(f * v.x, f * v.y), sm100::pack_bf16(f * v.z, f * v.w));
    }
}

__device__ __forceinline__ uint32_t relu_bf16x2(uint32_t v) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&v);
    x = __hmax2(x, __float2bfloat162_rn(0.f));
    return *reinterpret_cast<uint32_t *>(&x);
}

// ---------------------------------------------------------------------------
// 3'. bf16, d = 64, fixed weights: step 3 with the global term on the tensor
// cores and the window in quarter-warps.  The block's Q rows (bf16, exact)
// times the bf16 image of Ubar (hi + lo terms, so the product keeps ~16
// significant bits) give Q_i Ubar; g_i = w_0 V_i + (Q_i Ubar) / (Q_i . s + eps).
// Then eight lanes per token, eight channels per lane: a row is one 16-byte
// load and a dot product three shuffles, four tokens per warp at a time.
// ---------------------------------------------------------------------------
constexpr int kQS = 72;   // row stride (bf16) of the staged Q rows and Ubar image: ldmatrix conflict-free

// Eight bf16 channels at `row` (16-byte aligned) as floats, optionally ReLU'd
// (on the packed pairs: max(x, 0) is exact in bf16).
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16 *row, float (&x)[8], bool relu) {
    uint4 w = *reinterpret_cast<const uint4 *>(row);
    if (relu) w = make_uint4(relu_bf16x2(w.x), relu_bf16x2(w.y), relu_bf16x2(w.z), relu_bf16x2(w.w));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = sm100::bf16_lo(u[k]);
        x[2 * k + 1] = sm100::bf16_hi(u[k]);
    }
}
// Sum over the eight lanes of a quarter-warp (lanes 8 q .. 8 q + 7).
__device__ __forceinline__ float group8_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}
__device__ __forceinline__ float dot8(const float (&x)[8], const float (&y)[8]) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) a = fmaf(x[k], y[k], a);
    return a;
}

__global__ void __launch_bounds__(kThreads, 4) bwd_token_a_tc(BwdProblem b) {
    constexpr int D = 64;
    using namespace sm100;
    __shared__ __align__(16) __nv_bfloat16 Ui[2 * D * kQS];   // Ubar hi rows a (cols e), then lo
    __shared__ __align__(16) __nv_bfloat16 Qs[kTpb * kQS];    // the block's Q rows (feature-mapped)
    __shared__ __align__(16) float G[kTpb][D + 4];            // Q_i Ubar
    __shared__ __align__(16) float s_sh[D];
    __shared__ float part[kWarps];
    const Problem &p = b.fwd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = blockIdx.x / b.nblk, blk = blockIdx.x % b.nblk;
    const int j0 = blk * kTpb, cnt = min(kTpb, p.n - j0);
    const size_t sbase = (size_t)sl * p.n * D;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(p.Q) + sbase;
    const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(p.K) + sbase;
    const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(p.V) + sbase;
    const __nv_bfloat16 *dO = static_cast<const __nv_bfloat16 *>(b.dO) + sbase;
    const float al = p.alpha[sl % p.heads], w0 = p.w[0];
    const float scale = 0.125f;   // 1 / sqrt(64)

    {
        const uint4 *img = reinterpret_cast<const uint4 *>(b.ubimg + (size_t)sl * 2 * D * D);
        for (int x = tid; x < 2 * D * 8; x += kThreads)
            *reinterpret_cast<uint4 *>(Ui + (x >> 3) * kQS + (x & 7) * 8) = img[x];
        for (int x = tid; x < kTpb * 8; x += kThreads) {
            const int j = x >> 3, c = x & 7;
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (j < cnt) {
                q = reinterpret_cast<const uint4 *>(Q)[((size_t)(j0 + j) * D) / 8 + c];
                if (p.relu) q = make_uint4(relu_bf16x2(q.x), relu_bf16x2(q.y), relu_bf16x2(q.z), relu_bf16x2(q.w));
            }
            *reinterpret_cast<uint4 *>(Qs + j * kQS + c * 8) = q;
        }
        if (tid < D) s_sh[tid] = p.s_red[(size_t)sl * D + tid];
    }
    __syncthreads();

    // ---- Q Ubar: warp = 16 tokens (mt) x 16 columns (sb), hi and lo terms
    {
        const int mt = warp & 1, sb = warp >> 1;
        const uint32_t ua = smem_u32(Ui), qa = smem_u32(Qs);
        const int arow = 16 * mt + (lane & 15), acol = (lane >> 4) * 8;
        const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7), bcol = 16 * sb + (mi >> 1) * 8;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(qa + (uint32_t)(arow * kQS + 16 * ks + acol) * 2u, a0, a1, a2, a3);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(ua + (uint32_t)((h * D + 16 * ks + brow) * kQS + bcol) * 2u, b0, b1, b2, b3);
                mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(acc[1], a0, a1, a2, a3, b2, b3);
            }
        }
        const int row = 16 * mt + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int col = 16 * sb + 8 * nt + 2 * (lane & 3);
            G[row][col] = acc[nt][0];
            G[row][col + 1] = acc[nt][1];
            G[row + 8][col] = acc[nt][2];
            G[row + 8][col + 1] = acc[nt][3];
        }
    }
    __syncthreads();

    // ---- quarter-warp per token: window softmax statistics, dl . l, dalpha terms
    const int qg = lane >> 3, c8 = 8 * (lane & 7);
    const int u = 4 * warp + qg;              // this quarter's token in the block
    const bool live = u < cnt;
    const int i = live ? j0 + u : j0;         // dead quarters repeat a valid token; nothing is kept
    float q[8], v[8], go[8], g[8], sv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        q[k] = __bfloat162float(Qs[u * kQS + c8 + k]);
        sv[k] = s_sh[c8 + k];
    }
    load8_bf16(V + (size_t)i * D + c8, v, false);
    load8_bf16(dO + (size_t)i * D + c8, go, false);
    const float rq = 1.f / (group8_sum(dot8(q, sv)) + p.eps);
#pragma unroll
    for (int k = 0; k < 8; ++k) g[k] = fmaf(rq, G[u][c8 + k], w0 * v[k]);
    // the 3 x 3 window in row-major order; neighbours off the grid are masked
    const int r = i / p.W, c = i % p.W;
    float e[9];
#pragma unroll
    for (int t9 = 0; t9 < 9; ++t9) {
        const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
        const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
        float kr[8];
        load8_bf16(K + (size_t)(in ? rr * p.W + cc : i) * D + c8, kr, p.relu);
        e[t9] = dot8(q, kr);
    }
#pragma unroll
    for (int t9 = 0; t9 < 9; ++t9) e[t9] = group8_sum(e[t9]);
    float emax = -INFINITY;
#pragma unroll
    for (int t9 = 0; t9 < 9; ++t9) {
        const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
        const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
        e[t9] = in ? e[t9] * scale : -INFINITY;
        emax = fmaxf(emax, e[t9]);
    }
    float l[8], esum = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) l[k] = 0.f;
#pragma unroll
    for (int t9 = 0; t9 < 9; ++t9) {
        const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
        const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
        const float a = in ? ex2_approx((e[t9] - emax) * 1.4426950408889634f) : 0.f;   // as the tiled pass
        esum += a;
        float vr[8];
        load8_bf16(V + (size_t)(in ? rr * p.W + cc : i) * D + c8, vr, false);
#pragma unroll
        for (int k = 0; k < 8; ++k) l[k] = fmaf(a, vr[k], l[k]);
    }
    const float inv = 1.f / esum;
    float dgl = 0.f, dll = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        l[k] *= inv;
        dgl = fmaf(go[k], g[k] - l[k], dgl);
        dll = fmaf(go[k], l[k], dll);
    }
    dgl = group8_sum(dgl);
    dll = group8_sum(dll) * (1.f - al);
    if ((lane & 7) == 0 && live)
        reinterpret_cast<float4 *>(b.lstat)[(size_t)sl * p.n + j0 + u] = make_float4(emax, esum, dll, 0.f);
    // dalpha terms of the warp's live tokens, in token order
    float dal = ((lane & 7) == 0 && live) ? dgl : 0.f;
    dal = warp_sum(dal);
    if (lane == 0) part[warp] = dal;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int w = 0; w < kWarps; ++w) acc += part[w];
        b.dal_part[(size_t)sl * b.nblk + blk] = acc;
    }
}

// ---------------------------------------------------------------------------
// 5''. bf16, d = 64, fixed weights: the token pass on 8 x 8 token tiles.  A
// persistent CTA of 16 warps walks a contiguous run of tiles.  Each tile's
// halo (10 x 10 grid positions) of K, V, Q (feature-mapped) and dO, and the
// halo tokens' window statistics, arrive in shared memory by TMA (tiled 4-D
// boxes, zero-filled off the grid; 128-byte swizzled rows) while the
// previous tile computes (two halo buffers); the three d x d products gather
// their A rows from the halo (ldmatrix takes a row address per lane).
// ---------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kHaloSide = 10;                 // an 8 x 8 tile and its one-token border
constexpr int kHaloRows = kHaloSide * kHaloSide;
constexpr int kTileTok = 64;
constexpr int kTileWarps = 16;
constexpr int kTileThreads = 32 * kTileWarps;
// one halo buffer: K, V, Q, dO as 100 rows of 128 B each (a 1024-byte
// multiple apart, as the 128-byte swizzle wants), then the 100 statistics
constexpr int kHaloTensor = (kHaloRows * 128 + 1023) / 1024 * 1024;
constexpr int kHaloStats = 4 * kHaloTensor;
constexpr int kHaloBytes = (kHaloStats + kHaloRows * 16 + 1023) / 1024 * 1024;
constexpr uint32_t kHaloTx = 4u * kHaloRows * 128u + kHaloRows * 16u;     // bytes one tile's TMA delivers
constexpr int kOS = 68;                      // row stride (floats) of the products' outputs: conflict-free column reads
constexpr int kTileSmemBytes =
    1024 + 2 * kHaloBytes + kImgRows * kBS * 2 + kTileTok * kQS * 2 + 3 * kTileTok * kOS * 4;

// Halo row of the grid position (dy, dx) away from the tile's token u.
__device__ __forceinline__ int halo_row(int u, int dy, int dx) {
    return (u / 8 + 1 + dy) * kHaloSide + (u % 8 + 1 + dx);
}
// Byte offset of 16-byte chunk `chunk` of halo row `row` (128-byte swizzle).
__device__ __forceinline__ uint32_t hoff(int row, int chunk) {
    return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}
// Eight bf16 channels (chunk `chunk`) of halo row `row` as floats.
__device__ __forceinline__ void lds8_sw(const uint8_t *region, int row, int chunk, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4 *>(region + hoff(row, chunk));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = sm100::bf16_lo(u[k]);
        x[2 * k + 1] = sm100::bf16_hi(u[k]);
    }
}

template <bool kMlp>
__global__ void __launch_bounds__(kTileThreads, 1)
    bwd_token_b_tile(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                     const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mG,
                     const __grid_constant__ CUtensorMap mL, BwdProblem b) {
    constexpr int D = 64;
    using namespace sm100;
    extern __shared__ uint8_t smem_tile_raw[];
    uint8_t *halo0 = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_tile_raw) + 1023) & ~uintptr_t(1023));
    __nv_bfloat16 *Bs = reinterpret_cast<__nv_bfloat16 *>(halo0 + 2 * kHaloBytes);
    __nv_bfloat16 *Qt = Bs + kImgRows * kBS;   // Q~ of the tile's tokens
    __shared__ __align__(8) uint64_t hbar[2];   // a halo buffer's TMA landed
    float *oQ = reinterpret_cast<float *>(Qt + kTileTok * kQS), *oV = oQ + kTileTok * kOS, *oK = oV + kTileTok * kOS;
    __shared__ float rqs[kTileTok];
    __shared__ float cjs[kTileTok];
    __shared__ float dsw[kTileWarps][D];
    __shared__ float wts_t[kMlp ? kTileTok : 1][kMlp ? LISA_MAX_T_MLP : 1];   // adaptive weights of the tile's tokens
    const Problem &p = b.fwd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tiles_c = (p.W + 7) / 8;
    const long long ntiles = (long long)p.slices * b.ntile;
    const int t_begin = (int)(blockIdx.x * ntiles / gridDim.x), t_end = (int)((blockIdx.x + 1) * ntiles / gridDim.x);
    const float scale = 0.125f;   // 1 / sqrt(64)
    const int qg = lane >> 3, c8 = 8 * (lane & 7);
    const int u = 4 * warp + qg;   // this quarter's token of a tile

    if (tid == 0) {
        mbar_init(smem_u32(&hbar[0]), 1);
        mbar_init(smem_u32(&hbar[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the halo of tile t (K, V, Q, dO rows, statistics) into buffer `buf`; one thread
    auto stage_halo = [&](int t, int buf) {
        const int sl = t / b.ntile, tile = t % b.ntile;
        const int r0 = (tile / tiles_c) * 8, c0 = (tile % tiles_c) * 8;
        const uint32_t hb = smem_u32(halo0 + buf * kHaloBytes), bar = smem_u32(&hbar[buf]);
        fence_proxy_async();   // this buffer's earlier generic writes (the ReLU pass) before the async ones
        mbar_arrive_expect_tx(bar, kHaloTx);
        tma_load_4d(hb, &mK, 0, c0 - 1, r0 - 1, sl, bar);
        tma_load_4d(hb + kHaloTensor, &mV, 0, c0 - 1, r0 - 1, sl, bar);
        tma_load_4d(hb + 2 * kHaloTensor, &mQ, 0, c0 - 1, r0 - 1, sl, bar);
        tma_load_4d(hb + 3 * kHaloTensor, &mG, 0, c0 - 1, r0 - 1, sl, bar);
        tma_load_4d(hb + kHaloStats, &mL, 0, c0 - 1, r0 - 1, sl, bar);
    };

    int img_sl = -1;
    if (t_begin < t_end && tid == 0) stage_halo(t_begin, 0);
    for (int t = t_begin, it = 0; t < t_end; ++t, ++it) {
        const int cur = it & 1;
        // the next tile's halo streams in while this one computes; its buffer
        // was last read by the tile before this one, which ended on a barrier
        if (t + 1 < t_end && tid == 0) stage_halo(t + 1, cur ^ 1);
        float wpre = 0.f;   // adaptive weights: this thread's w of the tile, in flight during the halo wait
        if (kMlp && tid < kTileTok * p.T) {
            const int tsl = t / b.ntile, ttile = t % b.ntile, uu = tid / p.T;
            const int rr = (ttile / tiles_c) * 8 + uu / 8, cc = (ttile % tiles_c) * 8 + uu % 8;
            if (rr < p.H && cc < p.W) wpre = b.wtok[((size_t)tsl * p.n + rr * p.W + cc) * p.T + tid % p.T];
        }
        if (!mbar_wait(smem_u32(&hbar[cur]), (uint32_t)(it >> 1) & 1u)) record_error(p.err, kErrTimeoutLoad);
        const int sl = t / b.ntile, tile = t % b.ntile;
        const int r0 = (tile / tiles_c) * 8, c0 = (tile % tiles_c) * 8;
        if (sl != img_sl) {   // the slice's B image (tiles of one slice are consecutive)
            const uint4 *img = reinterpret_cast<const uint4 *>(b.bimg + (size_t)sl * kImgRows * D);
            for (int x = tid; x < kImgRows * 8; x += kTileThreads)
                *reinterpret_cast<uint4 *>(Bs + (x >> 3) * kBS + (x & 7) * 8) = img[x];
            img_sl = sl;
        }
        __syncthreads();   // the B image is in place
        uint8_t *Kc = halo0 + cur * kHaloBytes;
        uint8_t *Vc = Kc + kHaloTensor, *Qc = Kc + 2 * kHaloTensor, *Gc = Kc + 3 * kHaloTensor;
        const float4 *Lc = reinterpret_cast<const float4 *>(Kc + kHaloStats);
        if (p.relu) {   // the feature map of K and Q, in place (layout-blind: every 16-byte chunk)
            for (int x = tid; x < 2 * kHaloRows * 8; x += kTileThreads) {
                uint8_t *base = x < kHaloRows * 8 ? Kc : Qc;
                const int y = x % (kHaloRows * 8);
                uint4 *pv = reinterpret_cast<uint4 *>(base + y * 16);
                const uint4 v = *pv;
                *pv = make_uint4(relu_bf16x2(v.x), relu_bf16x2(v.y), relu_bf16x2(v.z), relu_bf16x2(v.w));
            }
            __syncthreads();
        }
        const size_t sbase = (size_t)sl * p.n * D;
        __nv_bfloat16 *dQo = static_cast<__nv_bfloat16 *>(b.dQ) + sbase;
        __nv_bfloat16 *dVo = static_cast<__nv_bfloat16 *>(b.dV) + sbase;
        float *dKp = b.dk_part + sbase;
        const float *s = p.s_red + (size_t)sl * D;
        const float al = p.alpha[sl % p.heads], w0 = p.w[0];
        {   // 1 / (Q_u . s + eps) and Q~_u (bf16) for the second product
            float q[8], sv[8];
            lds8_sw(Qc, halo_row(u, 0, 0), c8 >> 3, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) sv[e] = s[c8 + e];
            const float rq = 1.f / (group8_sum(dot8(q, sv)) + p.eps);
            if ((lane & 7) == 0) rqs[u] = rq;
            *reinterpret_cast<uint4 *>(Qt + u * kQS + c8) =
                make_uint4(pack_bf16(q[0] * rq, q[1] * rq), pack_bf16(q[2] * rq, q[3] * rq),
                           pack_bf16(q[4] * rq, q[5] * rq), pack_bf16(q[6] * rq, q[7] * rq));
        }
        if (kMlp && tid < kTileTok * p.T) wts_t[tid / p.T][tid % p.T] = wpre;   // 0 off the grid
        __syncthreads();

        // ---- the three products: warp = 16 tokens (mt) x 16 columns (sb) of each
        //   dQ~ = [dO | K] [alpha Ubar^T ; dM],  dK = [V | Q~] [dU_1^T ; dM^T],  dV = K dU_1
        // (adaptive weights: the image holds alpha U_1^T where alpha Ubar^T stands, and
        // the dO half of dQ~'s sum is scaled by each token's own w_1)
        {
            const int mt = warp & 3, sb = warp >> 2;
            const int ua = 16 * mt + (lane & 15), acol = (lane >> 4) * 8;
            const int hrow = halo_row(ua, 0, 0);
            const uint32_t trow = (uint32_t)ua * kQS;
            const uint32_t bs = smem_u32(Bs);
            const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7), bcol = 16 * sb + (mi >> 1) * 8;
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
                const int brow0 = pr == 0 ? 0 : (pr == 1 ? 128 : 256);
                const int ksteps = pr == 2 ? 4 : 8;
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float accw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // kMlp: dO U_1^T alpha
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    if (ks >= ksteps) break;
                    // A operand of this k-step: which halo row (or Q~ row), which 16 channels
                    const uint8_t *abuf = pr == 0 ? (ks < 4 ? Gc : Kc) : (pr == 1 ? Vc : Kc);
                    const uint32_t aaddr = (pr == 1 && ks >= 4)
                                               ? smem_u32(Qt) + (trow + 16 * (ks & 3) + acol) * 2u
                                               : smem_u32(abuf) + hoff(hrow, 2 * (ks & 3) + (lane >> 4));
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldsm_x4(aaddr, a0, a1, a2, a3);
                    ldsm_x4_t(bs + (uint32_t)((brow0 + 16 * ks + brow) * kBS + bcol) * 2u, b0, b1, b2, b3);
                    if (kMlp && pr == 0 && ks < 4) {
                        mma_bf16_16816(accw[0], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(accw[1], a0, a1, a2, a3, b2, b3);
                    } else {
                        mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(acc[1], a0, a1, a2, a3, b2, b3);
                    }
                }
                float *out = pr == 0 ? oQ : (pr == 1 ? oK : oV);
                const int row = 16 * mt + (lane >> 2);
                if (kMlp && pr == 0) {
                    const float w1a = p.T > 1 ? wts_t[row][1] : 0.f, w1b = p.T > 1 ? wts_t[row + 8][1] : 0.f;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        acc[nt][0] = fmaf(w1a, accw[nt][0], acc[nt][0]);
                        acc[nt][1] = fmaf(w1a, accw[nt][1], acc[nt][1]);
                        acc[nt][2] = fmaf(w1b, accw[nt][2], acc[nt][2]);
                        acc[nt][3] = fmaf(w1b, accw[nt][3], acc[nt][3]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 16 * sb + 8 * nt + 2 * (lane & 3);
                    out[row * kOS + col] = acc[nt][0];
                    out[row * kOS + col + 1] = acc[nt][1];
                    out[(row + 8) * kOS + col] = acc[nt][2];
                    out[(row + 8) * kOS + col + 1] = acc[nt][3];
                }
            }
        }
        if (kMlp && p.T > 2) {
            // ---- adaptive weights: the walk terms of k >= 2, dQ~_u += alpha w_uk dO_u U_k^T,
            // as dO U_k^T on mma.sync per k (alpha U_k^T's bf16 image staged where Q~ was,
            // which the products no longer read), each row scaled by its token's w_uk
            const int mt = warp & 3, sb = warp >> 2;
            const int hrow = halo_row(16 * mt + (lane & 15), 0, 0);
            const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7), bcol = 16 * sb + (mi >> 1) * 8;
            const int row = 16 * mt + (lane >> 2);
            for (int kk = 2; kk < p.T; ++kk) {
                __syncthreads();   // the products (or the previous k) no longer read the Q~ region
                const uint4 *img =
                    reinterpret_cast<const uint4 *>(b.ukimgT + ((size_t)sl * b.nh + (kk - 1)) * 64 * kQS);
                for (int x = tid; x < 64 * kQS / 8; x += kTileThreads) reinterpret_cast<uint4 *>(Qt)[x] = img[x];
                __syncthreads();
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                    ldsm_x4(smem_u32(Gc) + hoff(hrow, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
                    ldsm_x4_t(smem_u32(Qt) + (uint32_t)((16 * ks + brow) * kQS + bcol) * 2u, b0, b1, b2, b3);
                    mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(acc[1], a0, a1, a2, a3, b2, b3);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float wk = wts_t[row + 8 * h][kk];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = 16 * sb + 8 * nt + 2 * (lane & 3);
                        float *o = oQ + (row + 8 * h) * kOS + col;
                        o[0] = fmaf(wk, acc[nt][2 * h], o[0]);
                        o[1] = fmaf(wk, acc[nt][2 * h + 1], o[1]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- per token (quarter-warp): the normaliser's cj = (dQ~_u . Q_u) rq^2 and the ds terms
        {
            float dsl[8];
            const int y = u / 8, xx = u % 8;
            const bool live = r0 + y < p.H && c0 + xx < p.W;
            float4 xm[4];   // adaptive weights: the MLP's share of [dq | dk] for these channels
            if (kMlp && live) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    b.dxm + ((size_t)sl * p.n + (r0 + y) * p.W + c0 + xx) * 2 * D + c8);
                xm[0] = src[0], xm[1] = src[1], xm[2] = src[16], xm[3] = src[17];
            }
            float q[8], dqt[8];
            lds8_sw(Qc, halo_row(u, 0, 0), c8 >> 3, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) dqt[e] = oQ[u * kOS + c8 + e];
            const float rq = rqs[u];
            const float cj = group8_sum(dot8(dqt, q)) * rq * rq;
            if ((lane & 7) == 0) cjs[u] = cj;
            if (kMlp && live) {   // oQ becomes dq before the window term (dQ~ rq - cj s + the MLP's dq), oK gains dk
                const float xq[8] = {xm[0].x, xm[0].y, xm[0].z, xm[0].w, xm[1].x, xm[1].y, xm[1].z, xm[1].w};
                const float xk[8] = {xm[2].x, xm[2].y, xm[2].z, xm[2].w, xm[3].x, xm[3].y, xm[3].z, xm[3].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    oQ[u * kOS + c8 + e] = dqt[e] * rq - cj * s[c8 + e] + xq[e];
                    oK[u * kOS + c8 + e] += xk[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) dsl[e] = live ? -cj * q[e] : 0.f;
            // the warp's four tokens' ds terms, summed over the quarters in a fixed order
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                dsl[e] += __shfl_xor_sync(0xffffffffu, dsl[e], 8);
                dsl[e] += __shfl_xor_sync(0xffffffffu, dsl[e], 16);
            }
            if (qg == 0)
#pragma unroll
                for (int e = 0; e < 8; ++e) dsw[warp][c8 + e] = dsl[e];
        }
        __syncthreads();

        // ---- the window on the tensor cores: warp = block beta (tile rows 2 beta,
        // 2 beta + 1) x role (0: the block's tokens as queries -> dQ; 1: as keys
        // -> dK; 2: as keys -> dV).  Scores of the 16 tokens against the 4 x 10
        // window of the block; only the 3 x 3 window of each token counts.
        const int beta = warp & 3, role = warp >> 2;
        if (role < 3) {
            const int g = lane >> 2, q4 = lane & 3;
            // halo row of the block's fragment row m, and of window position kappa
            auto hrow_b = [&](int m) { return (2 * beta + 1 + (m >> 3)) * kHaloSide + (m & 7) + 1; };
            auto hrow_w = [&](int kappa) { return (2 * beta + kappa / 10) * kHaloSide + kappa % 10; };
            // bit j*4+e: window position 8j + 2 q4 + (e & 1) is inside the 3 x 3 window of
            // fragment row g + 8 (e >> 1) and inside the grid
            uint32_t wmask = 0;
#pragma unroll
            for (int j = 0; j < 5; ++j)
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int kappa = 8 * j + 2 * q4 + bb, ka = kappa / 10, kb = kappa % 10;
                    const int gr = r0 - 1 + 2 * beta + ka, gc = c0 - 1 + kb;
                    if (gr < 0 || gr >= p.H || gc < 0 || gc >= p.W) continue;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int du = ka - h, dv = kb - g;
                        if (du >= 0 && du <= 2 && dv >= 0 && dv <= 2) wmask |= 1u << (j * 4 + 2 * h + bb);
                    }
                }
            const uint32_t arow_m = (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1));   // A-fragment row of this lane
            // scores [16 x 40] = rows(Ab) . rows(Bw)^T over the 64 channels
            auto scores = [&](const uint8_t *Ab, const uint8_t *Bw, float (&sc)[5][4]) {
#pragma unroll
                for (int j = 0; j < 5; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                const int ar = hrow_b(arow_m);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(smem_u32(Ab) + hoff(ar, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                    for (int pr = 0; pr < 3; ++pr) {
                        const int kk = 8 * (2 * pr + (lane >> 4)) + (lane & 7);
                        const int kk2 = kk < 40 ? kk : 0;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(smem_u32(Bw) + hoff(hrow_w(kk2), 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
                        mma_bf16_16816(sc[2 * pr], a0, a1, a2, a3, b0, b1);
                        if (pr < 2) mma_bf16_16816(sc[2 * pr + 1], a0, a1, a2, a3, b2, b3);
                    }
                }
            };
            // acc [16 x 64] = w [16 x 40] . rows(Xw) (w in C-fragment layout, rounded to bf16)
            auto times_window = [&](const float (&w)[5][4], const uint8_t *Xw, float (&acc)[8][4]) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 3; ++ks) {
                    const int j0 = 2 * ks, j1 = 2 * ks + 1;
                    const uint32_t pa0 = pack_bf16(w[j0][0], w[j0][1]), pa1 = pack_bf16(w[j0][2], w[j0][3]);
                    const uint32_t pa2 = j1 < 5 ? pack_bf16(w[j1][0], w[j1][1]) : 0u;
                    const uint32_t pa3 = j1 < 5 ? pack_bf16(w[j1][2], w[j1][3]) : 0u;
                    const int kv = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
                    const int vr = hrow_w(kv < 40 ? kv : 0);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(Xw) + hoff(vr, 2 * np + (lane >> 4)), b0, b1, b2, b3);
                        mma_bf16_16816(acc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
                        mma_bf16_16816(acc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
                    }
                }
            };
            float sc[5][4], acc[8][4];
            if (role == 0) {
                // the block's tokens as queries: P = softmax weights (their own statistics),
                // dP = dl_i . V_j, de = P (dP - dl_i . l_i) / sqrt(d); dQ window term = de K
                scores(Qc, Kc, sc);
                float emx[2], ies[2], dll[2];   // row statistics, the max in log2 units
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 sh = Lc[hrow_b(g + 8 * h)];
                    emx[h] = sh.x * kLog2e;
                    ies[h] = 1.f / sh.y;
                    dll[h] = sh.z;
                }
                float dp[5][4];
                scores(Gc, Vc, dp);
#pragma unroll
                for (int j = 0; j < 5; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const float a = ((wmask >> (j * 4 + e)) & 1u)
                                            ? ex2_approx(fmaf(sc[j][e], scale * kLog2e, -emx[h])) * ies[h] : 0.f;
                        sc[j][e] = a * (dp[j][e] * (1.f - al) - dll[h]) * scale;
                    }
                times_window(sc, Kc, acc);
            } else {
                // the block's tokens as keys of the window's queries: P' with each query's
                // statistics; role 1: de' = P' (dP' - dl_i . l_i) / sqrt(d), dK term = de' Q;
                // role 2: dV term = (1 - alpha) P' dO
                scores(Kc, Qc, sc);
                float dp[5][4];
                if (role == 1) scores(Vc, Gc, dp);
#pragma unroll
                for (int j = 0; j < 5; ++j)
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        const int kappa = 8 * j + 2 * q4 + bb;
                        const float4 sk = Lc[hrow_w(kappa < 40 ? kappa : 0)];
                        const float emx = sk.x * kLog2e, ies = ((wmask >> (j * 4 + bb)) & 0x5u) ? 1.f / sk.y : 0.f;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int e = 2 * h + bb;
                            const float a = ((wmask >> (j * 4 + e)) & 1u)
                                                ? ex2_approx(fmaf(sc[j][e], scale * kLog2e, -emx)) * ies : 0.f;
                            sc[j][e] = role == 1 ? a * (dp[j][e] * (1.f - al) - sk.z) * scale : a * (1.f - al);
                        }
                    }
                times_window(sc, role == 1 ? Qc : Gc, acc);
            }
            // ---- combine with the products' terms and store (C-fragment layout)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = g + 8 * h, ut = (2 * beta + h) * 8 + g;   // tile token of fragment row m
                const int rr = r0 + 2 * beta + h, cc = c0 + g;
                if (rr >= p.H || cc >= p.W) continue;
                const size_t jt = (size_t)(rr * p.W + cc) * D;
                const float rq = rqs[ut], cj = cjs[ut];
                const float wv0 = kMlp ? wts_t[ut][0] : w0;   // adaptive weights: the token's own w_0
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int col = 8 * nt + 2 * q4;
                    const float x0 = acc[nt][2 * h], x1 = acc[nt][2 * h + 1];
                    if (role == 0) {
                        // (adaptive weights: oQ already holds dq before the window term)
                        float d0 = kMlp ? oQ[ut * kOS + col] + x0 : oQ[ut * kOS + col] * rq - cj * s[col] + x0;
                        float d1 = kMlp ? oQ[ut * kOS + col + 1] + x1
                                        : oQ[ut * kOS + col + 1] * rq - cj * s[col + 1] + x1;
                        if (p.relu) {   // dXq through the feature map (the staged Q is ReLU'd)
                            const uint32_t qp =
                                *reinterpret_cast<const uint32_t *>(Qc + hoff(hrow_b(m), col >> 3) + (col & 7) * 2);
                            if (!(bf16_lo(qp) > 0.f)) d0 = 0.f;
                            if (!(bf16_hi(qp) > 0.f)) d1 = 0.f;
                        }
                        *reinterpret_cast<uint32_t *>(dQo + jt + col) = pack_bf16(d0, d1);
                    } else if (role == 1) {
                        *reinterpret_cast<float2 *>(dKp + jt + col) =
                            make_float2(oK[ut * kOS + col] + x0, oK[ut * kOS + col + 1] + x1);
                    } else {
                        const uint32_t gp =
                            *reinterpret_cast<const uint32_t *>(Gc + hoff(hrow_b(m), col >> 3) + (col & 7) * 2);
                        const float d0 = fmaf(wv0 * al, bf16_lo(gp), oV[ut * kOS + col]) + x0;
                        const float d1 = fmaf(wv0 * al, bf16_hi(gp), oV[ut * kOS + col + 1]) + x1;
                        *reinterpret_cast<uint32_t *>(dVo + jt + col) = pack_bf16(d0, d1);
                    }
                }
            }
        }
        __syncthreads();
        for (int ch = tid; ch < D; ch += kTileThreads) {
            float acc = 0.f;
            for (int w = 0; w < kTileWarps; ++w) acc += dsw[w][ch];
            b.ds_part[((size_t)sl * b.ntile + tile) * D + ch] = acc;
        }
        __syncthreads();   // every read of this tile's buffers, Qt, the outputs and dsw is done
    }
}

// ---------------------------------------------------------------------------
// 3a'. bf16, d = 64, adaptive weights: step 3a with its three products on the
// tensor cores, per block of 32 tokens (mma.sync, bf16 operands, fp32
// accumulation; W1, U_k and da enter as bf16 hi + lo terms, Q and K are exact
// in bf16): the hidden pre-activations [Q | K] W1^T, the walk terms
// Y_k = Q U_k (k = 1 .. T-1, one U_k image at a time, folded into g and the
// dw partials as they come out), and the MLP's share of [dq; dk] = da W1.
// The softmax, the window and the MLP's elementwise backward stay per token.
// ---------------------------------------------------------------------------
constexpr int kMA = 136;                 // [Q | K] and W1 image row stride (bf16): 128 channels + pad
constexpr int kMH = LISA_MAX_HIDDEN;     // hidden units held (a multiple of 16)
constexpr int kMlpTcSmemBytes = kTpb * kMA * 2              // [Q | K] rows
                                + 2 * kMH * kMA * 2         // W1 hi, lo
                                + 2 * 64 * kQS * 2          // U_k hi, lo
                                + 2 * kTpb * kQS * 2        // da hi, lo
                                + 3 * kTpb * 68 * 4         // pre-activations (then da), g, V and dO rows (fp32)
                                + kTpb * 68 * 4;

// The tensor-core MLP passes' bf16 operand images, once per backward: block
// (slice, k) writes U_k (row-major) as hi and lo rows of kQS columns and
// alpha U_k^T (row c, column a) rounded to bf16, the last block W1 as hi and lo
// rows of kMA columns (rows hidden .. kMH - 1 zero).
__global__ void __launch_bounds__(kThreads) bwd_mlp_images(BwdProblem b) {
    constexpr int D = 64;
    const Problem &p = b.fwd;
    const int tid = threadIdx.x;
    if (blockIdx.x < (unsigned)(p.slices * b.nh)) {
        const float *Ut = b.Uk + (size_t)blockIdx.x * D * D;   // transposed: Ut[e * D + a] = U_k[a][e]
        uint16_t *img = b.ukimg + (size_t)blockIdx.x * 2 * 64 * kQS;
        uint16_t *imgT = b.ukimgT + (size_t)blockIdx.x * 64 * kQS;
        const float al = p.alpha[(blockIdx.x / b.nh) % p.heads];
        __shared__ float tile[D][D + 1];   // tile[e][a] = U_k[a][e]; both images written row by row
        for (int x = tid; x < D * D; x += kThreads) tile[x >> 6][x & 63] = Ut[x];
        __syncthreads();
        for (int x = tid; x < D * D; x += kThreads) {
            const int r = x >> 6, c = x & 63;
            imgT[r * kQS + c] = __bfloat16_as_ushort(__float2bfloat16_rn(al * tile[r][c]));
            const float uv = tile[c][r];   // U_k[r][c]
            const __nv_bfloat16 hi = __float2bfloat16_rn(uv);
            img[r * kQS + c] = __bfloat16_as_ushort(hi);
            img[64 * kQS + r * kQS + c] = __bfloat16_as_ushort(__float2bfloat16_rn(uv - __bfloat162float(hi)));
        }
    } else {
        for (int x = tid; x < kMH * 2 * D; x += kThreads) {
            const int m = x / (2 * D), c = x % (2 * D);
            const float w = m < p.hidden ? p.W1[(size_t)m * 2 * D + c] : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            b.w1img[m * kMA + c] = __bfloat16_as_ushort(hi);
            b.w1img[kMH * kMA + m * kMA + c] = __bfloat16_as_ushort(__float2bfloat16_rn(w - __bfloat162float(hi)));
        }
    }
}

__global__ void __launch_bounds__(kThreads) bwd_token_mlp_tc(BwdProblem b) {
    constexpr int D = 64, TM = LISA_MAX_T_MLP;
    using namespace sm100;
    extern __shared__ float4 smem_mlp[];
    __nv_bfloat16 *Qk = reinterpret_cast<__nv_bfloat16 *>(smem_mlp);   // [kTpb][kMA]: Q | K
    __nv_bfloat16 *W1i = Qk + kTpb * kMA;                              // [2][kMH][kMA]
    __nv_bfloat16 *Ui = W1i + 2 * kMH * kMA;                           // [2][64][kQS]
    __nv_bfloat16 *Di = Ui + 2 * 64 * kQS;                             // [2][kTpb][kQS]: da hi, lo
    float *pre = reinterpret_cast<float *>(Di + 2 * kTpb * kQS);      // [kTpb][68]
    float *G = pre + kTpb * 68;                                        // [kTpb][68]: g without w_0 V
    float *Vs = G + kTpb * 68;                                         // [kTpb][68]: V rows
    float *Gs = Vs + kTpb * 68;                                        // [kTpb][68]: dO rows
    __shared__ float rqs[kTpb];
    __shared__ float wts[kTpb][TM];
    __shared__ float dwp[TM][kTpb][4];    // dw_k partials per row and 16-column group
    __shared__ float part[kWarps];
    __shared__ float W2s[TM * kMH], b2s[TM];   // the MLP's second layer, staged once per CTA
    const Problem &p = b.fwd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.T, hid = p.hidden, nmh = (hid + 15) / 16 * 16;
    {   // W1 hi and lo rows from the precomputed image (the rows below nmh of each), once per CTA
        constexpr int kRowV = kMA / 8;   // 16-byte pieces per row
        const uint4 *img = reinterpret_cast<const uint4 *>(b.w1img);
        for (int x = tid; x < 2 * nmh * kRowV; x += kThreads) {
            const int h = x / (nmh * kRowV), y = x % (nmh * kRowV);
            reinterpret_cast<uint4 *>(W1i + h * kMH * kMA)[y] = img[h * kMH * kRowV + y];
        }
    }
    for (int x = tid; x < T * hid; x += kThreads) W2s[x] = p.W2[x];
    if (tid < T) b2s[tid] = p.b2[tid];
    // this thread's 16-byte piece of a block's Q, K, V and dO rows (token tid / 8,
    // channels 8 (tid % 8) ..), loaded one block ahead so the loads overlap the
    // previous block's work
    static_assert(kTpb * 8 == kThreads, "one 16-byte piece of each row per thread");
    uint4 rq_q, rq_k, rq_v, rq_g;
    auto load_rows = [&](int bj) {
        const int slj = bj / b.nblk, j0j = (bj % b.nblk) * kTpb, jj = tid >> 3;
        rq_q = rq_k = rq_v = rq_g = make_uint4(0u, 0u, 0u, 0u);
        if (j0j + jj < p.n) {
            const size_t o = ((size_t)slj * p.n * D + (size_t)(j0j + jj) * D) / 8 + (tid & 7);
            rq_q = reinterpret_cast<const uint4 *>(p.Q)[o];
            rq_k = reinterpret_cast<const uint4 *>(p.K)[o];
            rq_v = reinterpret_cast<const uint4 *>(p.V)[o];
            rq_g = reinterpret_cast<const uint4 *>(b.dO)[o];
        }
    };
    if (blockIdx.x < (unsigned)(p.slices * b.nblk)) load_rows(blockIdx.x);
    // persistent: the CTA walks blocks of kTpb tokens; W1 stays staged
    const int nbt = p.slices * b.nblk;
    for (int bi = blockIdx.x; bi < nbt; bi += gridDim.x) {
        const int sl = bi / b.nblk, blk = bi % b.nblk;
        const int j0 = blk * kTpb, cnt = min(kTpb, p.n - j0);
        const size_t sbase = (size_t)sl * p.n * D;
        const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(p.K) + sbase;   // the window's rows
        const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(p.V) + sbase;
        const float *s = p.s_red + (size_t)sl * D;
        const float al = p.alpha[sl % p.heads];

        // ---- stage [Q | K] (feature-mapped), V and dO rows (fp32) from the prefetched pieces
        {
            const int j = tid >> 3, c = tid & 7;
            uint4 q = rq_q, k = rq_k;
            const uint4 v = rq_v, g = rq_g;
            if (p.relu) {
                q = make_uint4(relu_bf16x2(q.x), relu_bf16x2(q.y), relu_bf16x2(q.z), relu_bf16x2(q.w));
                k = make_uint4(relu_bf16x2(k.x), relu_bf16x2(k.y), relu_bf16x2(k.z), relu_bf16x2(k.w));
            }
            *reinterpret_cast<uint4 *>(Qk + j * kMA + c * 8) = q;
            *reinterpret_cast<uint4 *>(Qk + j * kMA + 64 + c * 8) = k;
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w}, gg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                Vs[j * 68 + c * 8 + 2 * e] = bf16_lo(vv[e]);
                Vs[j * 68 + c * 8 + 2 * e + 1] = bf16_hi(vv[e]);
                Gs[j * 68 + c * 8 + 2 * e] = bf16_lo(gg[e]);
                Gs[j * 68 + c * 8 + 2 * e + 1] = bf16_hi(gg[e]);
            }
        }
        if (bi + (int)gridDim.x < nbt) load_rows(bi + (int)gridDim.x);   // the next block's rows, in flight
        for (int x = tid; x < TM * kTpb * 4; x += kThreads) (&dwp[0][0][0])[x] = 0.f;
        __syncthreads();
        for (int j = warp; j < kTpb; j += kWarps) {   // 1 / (Q_j . s + eps)
            float d = 0.f;
            for (int ch = lane; ch < D; ch += 32) d += __bfloat162float(Qk[j * kMA + ch]) * s[ch];
            d = warp_sum(d);
            if (lane == 0) rqs[j] = 1.f / (d + p.eps);
        }

        // ---- hidden pre-activations [Q | K] W1^T + b1: warp = 16 tokens x 16 hidden units
        {
            const int mt = warp & 1, pr = warp >> 1;   // n-tiles 2 pr, 2 pr + 1
            if (16 * pr < nmh) {
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const uint32_t qa = smem_u32(Qk) + (uint32_t)((16 * mt + (lane & 15)) * kMA + (lane >> 4) * 8) * 2u;
                const int wrow = 16 * pr + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(qa + (uint32_t)(16 * ks) * 2u, a0, a1, a2, a3);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t b0, b1, b2, b3;
                        const uint32_t wofs = (uint32_t)(h * kMH * kMA + wrow * kMA + 16 * ks + ((lane >> 3) & 1) * 8);
                        ldsm_x4(smem_u32(W1i) + wofs * 2u, b0, b1, b2, b3);
                        mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(acc[1], a0, a1, a2, a3, b2, b3);
                    }
                }
                const int row = 16 * mt + (lane >> 2);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int m = 16 * pr + 8 * nt + 2 * (lane & 3);
                    const float b10 = m < hid ? p.b1[m] : 0.f, b11 = m + 1 < hid ? p.b1[m + 1] : 0.f;
                    pre[row * 68 + m] = acc[nt][0] + b10;
                    pre[row * 68 + m + 1] = acc[nt][1] + b11;
                    pre[(row + 8) * 68 + m] = acc[nt][2] + b10;
                    pre[(row + 8) * 68 + m + 1] = acc[nt][3] + b11;
                }
            }
        }
        __syncthreads();
        // ---- per token (a quarter-warp, lanes over hidden units): h = GELU(a),
        // z = W2 h + b2, w = softmax(z)
        const int qg = lane >> 3, l8 = lane & 7;
        const int uq = 4 * warp + qg;   // this quarter's token of the block
        {
            float zt[TM];
#pragma unroll
            for (int t = 0; t < TM; ++t) zt[t] = 0.f;
            for (int m = l8; m < hid; m += 8) {
                const float h = gelu_as7126(pre[uq * 68 + m]);
#pragma unroll
                for (int t = 0; t < TM; ++t)
                    if (t < T) zt[t] = fmaf(W2s[t * hid + m], h, zt[t]);
                if (uq < cnt) b.hbuf[((size_t)sl * p.n + j0 + uq) * hid + m] = h;
            }
            float zmax = -INFINITY, zs = 0.f;
#pragma unroll
            for (int t = 0; t < TM; ++t)
                if (t < T) {
                    zt[t] = group8_sum(zt[t]) + b2s[t];
                    zmax = fmaxf(zmax, zt[t]);
                }
#pragma unroll
            for (int t = 0; t < TM; ++t)
                if (t < T) {
                    zt[t] = expf(zt[t] - zmax);
                    zs += zt[t];
                }
#pragma unroll
            for (int t = 0; t < TM; ++t)
                if (t < T && t == l8) wts[uq][t] = zt[t] / zs;
        }
        __syncthreads();

        // ---- walk terms Y_k = Q U_k on the tensor cores; g = sum_k w_k Y_k rq, and
        // dw_k partials alpha dO . Y_k rq per row and 16-column group
        {
            const int mt = warp & 1, sb = warp >> 1;
            const uint32_t qa = smem_u32(Qk) + (uint32_t)((16 * mt + (lane & 15)) * kMA + (lane >> 4) * 8) * 2u;
            const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7), bcol = 16 * sb + (mi >> 1) * 8;
            const int r0 = 16 * mt + (lane >> 2);
            float gacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int kk = 1; kk < T; ++kk) {
                {   // U_k's bf16 hi and lo rows from the precomputed image
                    const uint4 *img =
                        reinterpret_cast<const uint4 *>(b.ukimg + ((size_t)sl * b.nh + (kk - 1)) * 2 * 64 * kQS);
                    for (int x = tid; x < 2 * 64 * kQS / 8; x += kThreads) reinterpret_cast<uint4 *>(Ui)[x] = img[x];
                }
                __syncthreads();
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(qa + (uint32_t)(16 * ks) * 2u, a0, a1, a2, a3);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(Ui) + (uint32_t)((h * 64 + 16 * ks + brow) * kQS + bcol) * 2u, b0, b1, b2,
                                  b3);
                        mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(acc[1], a0, a1, a2, a3, b2, b3);
                    }
                }
                float dwr[2] = {0.f, 0.f};   // rows r0, r0 + 8
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = r0 + 8 * h;
                    const float rq = rqs[row], wk = wts[row][kk];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = 16 * sb + 8 * nt + 2 * (lane & 3);
                        const float y0 = acc[nt][2 * h] * rq, y1 = acc[nt][2 * h + 1] * rq;
                        gacc[nt][2 * h] = fmaf(wk, y0, gacc[nt][2 * h]);
                        gacc[nt][2 * h + 1] = fmaf(wk, y1, gacc[nt][2 * h + 1]);
                        dwr[h] = fmaf(Gs[row * 68 + col], y0, fmaf(Gs[row * 68 + col + 1], y1, dwr[h]));
                    }
                    dwr[h] += __shfl_xor_sync(0xffffffffu, dwr[h], 1);
                    dwr[h] += __shfl_xor_sync(0xffffffffu, dwr[h], 2);
                }
                if ((lane & 3) == 0) {
                    dwp[kk][r0][sb] = al * dwr[0];
                    dwp[kk][r0 + 8][sb] = al * dwr[1];
                }
                __syncthreads();   // every read of this U_k image is done
            }
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 16 * sb + 8 * nt + 2 * (lane & 3);
                    G[(r0 + 8 * h) * 68 + col] = gacc[nt][2 * h];
                    G[(r0 + 8 * h) * 68 + col + 1] = gacc[nt][2 * h + 1];
                }
        }
        __syncthreads();

        // ---- per token (a quarter-warp): the window (as bwd_token_a), dalpha terms,
        // the softmax's and the MLP's elementwise backward; da as bf16 hi + lo
        {
            const int c8 = 8 * l8;
            const bool live = uq < cnt;
            const int i = j0 + (live ? uq : 0);
            const int r = i / p.W, c = i % p.W;
            float q[8], v[8], go[8], g[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                q[e] = __bfloat162float(Qk[uq * kMA + c8 + e]);
                v[e] = Vs[uq * 68 + c8 + e];
                go[e] = Gs[uq * 68 + c8 + e];
                g[e] = fmaf(wts[uq][0], v[e], G[uq * 68 + c8 + e]);
            }
            float ev[9];
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
                const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
                float kr[8];
                load8_bf16(K + (size_t)(in ? rr * p.W + cc : i) * D + c8, kr, p.relu);
                ev[t9] = dot8(q, kr);
            }
            // the group sums run on every lane (each shuffle needs all 32); the mask after
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) ev[t9] = group8_sum(ev[t9]);
            float emax = -INFINITY;
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
                const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
                ev[t9] = in ? ev[t9] * 0.125f : -INFINITY;
                emax = fmaxf(emax, ev[t9]);
            }
            float l[8], esum = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) l[e] = 0.f;
#pragma unroll
            for (int t9 = 0; t9 < 9; ++t9) {
                const int rr = r + t9 / 3 - 1, cc = c + t9 % 3 - 1;
                const bool in = rr >= 0 && rr < p.H && cc >= 0 && cc < p.W;
                const float a = in ? ex2_approx((ev[t9] - emax) * 1.4426950408889634f) : 0.f;
                esum += a;
                float vr[8];
                load8_bf16(V + (size_t)(in ? rr * p.W + cc : i) * D + c8, vr, false);
#pragma unroll
                for (int e = 0; e < 8; ++e) l[e] = fmaf(a, vr[e], l[e]);
            }
            const float inv = 1.f / esum;
            float dgl = 0.f, dll = 0.f, dgv = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                l[e] *= inv;
                dgl = fmaf(go[e], g[e] - l[e], dgl);
                dll = fmaf(go[e], l[e], dll);
                dgv = fmaf(go[e], v[e], dgv);   // dw_0 / alpha
            }
            dgl = group8_sum(dgl);
            dll = group8_sum(dll);
            dgv = group8_sum(dgv);
            const size_t ti = (size_t)sl * p.n + i;
            if (l8 == 0 && live)
                reinterpret_cast<float4 *>(b.lstat)[ti] = make_float4(emax, esum, dll * (1.f - al), 0.f);
            // dz = w (dw - w . dw), dw_0 = alpha dO . V, dw_k from the partials
            float w[TM], dw[TM], wdw = 0.f;
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                w[t] = t < T ? wts[uq][t] : 0.f;
                dw[t] = t == 0 ? al * dgv
                               : (t < T ? ((dwp[t][uq][0] + dwp[t][uq][1]) + (dwp[t][uq][2] + dwp[t][uq][3])) : 0.f);
                wdw = fmaf(w[t], dw[t], wdw);
            }
            float dz[TM];
#pragma unroll
            for (int t = 0; t < TM; ++t) dz[t] = w[t] * (dw[t] - wdw);
            if (live) {
#pragma unroll
                for (int t = 0; t < TM; ++t)
                    if (t < T && t == l8) {
                        b.wtok[ti * T + t] = w[t];
                        b.dzbuf[ti * T + t] = dz[t];
                    }
            }
            for (int m = l8; m < nmh; m += 8) {
                float da = 0.f;
                if (m < hid && live) {
                    float dh = 0.f;
#pragma unroll
                    for (int t = 0; t < TM; ++t)
                        if (t < T) dh = fmaf(W2s[t * hid + m], dz[t], dh);
                    da = dh * gelu_grad_as7126(pre[uq * 68 + m]);
                    b.dabuf[ti * hid + m] = da;
                }
                const __nv_bfloat16 hi = __float2bfloat16_rn(da);
                Di[uq * kQS + m] = hi;
                Di[kTpb * kQS + uq * kQS + m] = __float2bfloat16_rn(da - __bfloat162float(hi));
            }
            // dalpha terms of the warp's live tokens, in token order
            float dal = (l8 == 0 && live) ? dgl : 0.f;
            dal = warp_sum(dal);
            if (lane == 0) part[warp] = dal;
        }
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
            for (int w2 = 0; w2 < kWarps; ++w2) acc += part[w2];
            b.dal_part[(size_t)sl * b.nblk + blk] = acc;
        }

        // ---- the MLP's share of [dq | dk] = da W1: warp = 16 tokens x 32 channels
        {
            const int mt = warp & 1, cg = warp >> 1;   // channels 32 cg .. 32 cg + 31
            const uint32_t da0 = smem_u32(Di) + (uint32_t)((16 * mt + (lane & 15)) * kQS + (lane >> 4) * 8) * 2u;
            const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7);
            float acc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            for (int ks = 0; 16 * ks < nmh; ++ks) {
#pragma unroll
                for (int ah = 0; ah < 2; ++ah) {   // da hi, lo
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(da0 + (uint32_t)(ah * kTpb * kQS + 16 * ks) * 2u, a0, a1, a2, a3);
#pragma unroll
                    for (int wh = 0; wh < 2; ++wh) {   // W1 hi, lo (lo x lo left out)
                        if (ah == 1 && wh == 1) continue;
#pragma unroll
                        for (int np = 0; np < 2; ++np) {
                            const int bcol = 32 * cg + 16 * np + (mi >> 1) * 8;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(smem_u32(W1i) + (uint32_t)(wh * kMH * kMA + (16 * ks + brow) * kMA + bcol) * 2u,
                                      b0, b1, b2, b3);
                            mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                            mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                        }
                    }
                }
            }
            const int row = 16 * mt + (lane >> 2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int u = row + 8 * h;
                if (u >= cnt) continue;
                float *xm = b.dxm + ((size_t)sl * p.n + j0 + u) * 2 * D;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int c = 32 * cg + 8 * nt + 2 * (lane & 3);
                    *reinterpret_cast<float2 *>(xm + c) = make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
                }
            }
        }
        __syncthreads();   // the next block restages the shared rows
    }
}

// ---------------------------------------------------------------------------
// 2'. adaptive weights on the tensor path (bf16, d = 64): the chunk's partial
// dU_k = sum_j Q_j (c_jk dO_j)^T with c_jk = alpha w_jk / (Q_j . s + eps), the
// same sum as bwd_stats_duk with the token's scalars moved onto dO.  Q^T is
// exact in bf16 (A operand, ldmatrix.trans from the token-major tile), c_jk dO_j
// goes in as bf16 hi + lo; one quarter-warp stages each token; a block takes
// kDukPerBlock walk lengths.
// ---------------------------------------------------------------------------
constexpr int kDukPerBlock = 2;   // walk lengths per block: Q and dO are staged once for both
__global__ void __launch_bounds__(kThreads) bwd_stats_duk_tc(BwdProblem b) {
    constexpr int D = 64, KP = kDukPerBlock;
    static_assert(kTpb * 8 == kThreads, "one quarter-warp per staged token");
    using namespace sm100;
    __shared__ __align__(16) __nv_bfloat16 Qs[kTpb][kQS];
    __shared__ __align__(16) __nv_bfloat16 Gs[KP][2][kTpb][kQS];   // per walk length: c dO hi, lo
    const Problem &p = b.fwd;
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, k0 = 1 + KP * blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(p.Q) + (size_t)sl * p.n * D;
    const __nv_bfloat16 *dO = static_cast<const __nv_bfloat16 *>(b.dO) + (size_t)sl * p.n * D;
    const float *wt = b.wtok + (size_t)sl * p.n * p.T;
    const float al = p.alpha[sl % p.heads];
    const int j8 = tid >> 3, c8 = tid & 7;   // staging: token j8, channels 8 c8 .. 8 c8 + 7
    float sv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) sv[u] = p.s_red[(size_t)sl * D + 8 * c8 + u];
    // warp: Q channels 16 mt .. 16 mt + 15 x dO channels 32 ng .. 32 ng + 31
    const int mt = warp & 3, ng = warp >> 2;
    const int arow = (lane & 7) + 8 * (lane >> 4), acol = 16 * mt + 8 * ((lane >> 3) & 1);
    const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7);
    float acc[KP][4][4];
#pragma unroll
    for (int kp = 0; kp < KP; ++kp)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) acc[kp][nt][0] = acc[kp][nt][1] = acc[kp][nt][2] = acc[kp][nt][3] = 0.f;
    for (int base = t0; base < t1; base += kTpb) {
        const bool in = j8 < t1 - base;
        float q[8], g[8];
        if (in) {
            load8_bf16(Q + (size_t)(base + j8) * D + 8 * c8, q, p.relu != 0);
            load8_bf16(dO + (size_t)(base + j8) * D + 8 * c8, g, false);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) q[u] = g[u] = 0.f;
        }
        const float den = group8_sum(dot8(q, sv)) + p.eps;   // every lane: the shuffles need all 32
        uint32_t qw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) qw[u] = pack_bf16(q[2 * u], q[2 * u + 1]);
        *reinterpret_cast<uint4 *>(&Qs[j8][8 * c8]) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
#pragma unroll
        for (int kp = 0; kp < KP; ++kp) {
            const int k = k0 + kp;
            const float cj = (in && k < p.T) ? al * wt[(size_t)(base + j8) * p.T + k] / den : 0.f;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float x0 = cj * g[2 * u], x1 = cj * g[2 * u + 1];
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                hw[u] = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                lw[u] = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
            }
            *reinterpret_cast<uint4 *>(&Gs[kp][0][j8][8 * c8]) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(&Gs[kp][1][j8][8 * c8]) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        __syncthreads();
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {   // tokens 16 ks .. 16 ks + 15
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(smem_u32(&Qs[16 * ks + arow][acol]), a0, a1, a2, a3);
#pragma unroll
            for (int kp = 0; kp < KP; ++kp)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(&Gs[kp][h][16 * ks + brow][32 * ng + 16 * np + (mi >> 1) * 8]), b0, b1,
                                  b2, b3);
                        mma_bf16_16816(acc[kp][2 * np], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(acc[kp][2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
        }
        __syncthreads();
    }
    const int g4 = lane >> 2, q4 = lane & 3;
#pragma unroll
    for (int kp = 0; kp < KP; ++kp) {
        const int k = k0 + kp;
        if (k >= p.T) break;
        float *out = b.dukp + (((size_t)sl * p.chunks + c) * b.nh + (k - 1)) * D * D;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                *reinterpret_cast<float2 *>(out + (size_t)(16 * mt + g4 + 8 * h) * D + 32 * ng + 8 * nt + 2 * q4) =
                    make_float2(acc[kp][nt][2 * h], acc[kp][nt][2 * h + 1]);
    }
}

// ---------------------------------------------------------------------------
// The MLP parameters' partial gradients per (slice, chunk), bf16 at d = 64:
// dW1 = sum_i da_i [q_i; k_i]^T on mma.sync over 32-token tiles (da as bf16
// hi + lo, its A fragments read from the token-major tile by ldmatrix.trans;
// [Q | K] exact in bf16), the small dW2 = sum_i dz_i h_i^T and the exact fp32
// sums db1, db2 on CUDA cores as in bwd_mlp_params.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 3) bwd_mlp_params_tc(BwdProblem b) {
    constexpr int D = 64;
    using namespace sm100;
    __shared__ __align__(16) __nv_bfloat16 Xs[kTpb][kMA];        // [Q | K] rows
    __shared__ __align__(16) __nv_bfloat16 Das[2][kTpb][kQS];    // da hi, lo (token-major)
    __shared__ float As[kTpb][LISA_MAX_HIDDEN];
    __shared__ float Hs[kTpb][LISA_MAX_HIDDEN];
    __shared__ float Zs[kTpb][LISA_MAX_T_MLP];
    const Problem &p = b.fwd;
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int T = p.T, hid = p.hidden, nmh = (hid + 15) / 16 * 16;
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const size_t sbase = (size_t)sl * p.n * D, tb = (size_t)sl * p.n;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(p.Q) + sbase;
    const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(p.K) + sbase;
    // warp: hidden rows 16 mt .. 16 mt + 15 x channels 64 ng .. 64 ng + 63
    const int mt = warp & 3, ng = warp >> 2;
    const bool mma_warp = 16 * mt < nmh;
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float w2[2] = {0.f, 0.f}, bb = 0.f;
    for (int base = t0; base < t1; base += kTpb) {
        const int cnt = min(kTpb, t1 - base);
        for (int x = tid; x < kTpb * 8; x += kThreads) {
            const int j = x >> 3, ch = x & 7;
            uint4 q = make_uint4(0u, 0u, 0u, 0u), k = q;
            if (j < cnt) {
                const size_t o = ((size_t)(base + j) * D) / 8 + ch;
                q = reinterpret_cast<const uint4 *>(Q)[o];
                k = reinterpret_cast<const uint4 *>(K)[o];
                if (p.relu) {
                    q = make_uint4(relu_bf16x2(q.x), relu_bf16x2(q.y), relu_bf16x2(q.z), relu_bf16x2(q.w));
                    k = make_uint4(relu_bf16x2(k.x), relu_bf16x2(k.y), relu_bf16x2(k.z), relu_bf16x2(k.w));
                }
            }
            *reinterpret_cast<uint4 *>(&Xs[j][ch * 8]) = q;
            *reinterpret_cast<uint4 *>(&Xs[j][64 + ch * 8]) = k;
        }
        for (int x = tid; x < kTpb * LISA_MAX_HIDDEN; x += kThreads) {
            const int j = x / LISA_MAX_HIDDEN, m = x % LISA_MAX_HIDDEN;
            const bool in = j < cnt && m < hid;
            const float da = in ? b.dabuf[(tb + base + j) * hid + m] : 0.f;
            As[j][m] = da;
            Hs[j][m] = in ? b.hbuf[(tb + base + j) * hid + m] : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(da);
            Das[0][j][m] = hi;
            Das[1][j][m] = __float2bfloat16_rn(da - __bfloat162float(hi));
        }
        for (int x = tid; x < kTpb * LISA_MAX_T_MLP; x += kThreads) {
            const int j = x / LISA_MAX_T_MLP, t = x % LISA_MAX_T_MLP;
            Zs[j][t] = (j < cnt && t < T) ? b.dzbuf[(tb + base + j) * T + t] : 0.f;
        }
        __syncthreads();
        if (mma_warp) {
            const int arow = (lane & 7) + 8 * (lane >> 4), acol = 16 * mt + 8 * ((lane >> 3) & 1);
            const int mi = lane >> 3, brow = (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {   // tokens 16 ks .. 16 ks + 15
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // da hi, lo
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(smem_u32(&Das[h][16 * ks + arow][acol]), a0, a1, a2, a3);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        const int bcol = 64 * ng + 16 * np + (mi >> 1) * 8;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(smem_u32(&Xs[16 * ks + brow][bcol]), b0, b1, b2, b3);
                        mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                        mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
                }
            }
        }
        for (int j = 0; j < cnt; ++j) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int e = tid + r * kThreads, t = e / LISA_MAX_HIDDEN, m = e % LISA_MAX_HIDDEN;
                if (t < LISA_MAX_T_MLP) w2[r] = fmaf(Zs[j][t], Hs[j][m], w2[r]);
            }
            if (tid < LISA_MAX_HIDDEN) bb += As[j][tid];
            else if (tid - LISA_MAX_HIDDEN < LISA_MAX_T_MLP) bb += Zs[j][tid - LISA_MAX_HIDDEN];
        }
        __syncthreads();
    }
    const size_t pc = (size_t)sl * p.chunks + c;
    if (mma_warp) {
        const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = 16 * mt + g + 8 * h;
            if (m >= hid) continue;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int ch = 64 * ng + 8 * nt + 2 * q4;
                *reinterpret_cast<float2 *>(b.pw1 + pc * hid * 2 * D + (size_t)m * 2 * D + ch) =
                    make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int e = tid + r * kThreads, t = e / LISA_MAX_HIDDEN, m = e % LISA_MAX_HIDDEN;
        if (t < T && m < hid) b.pw2[(pc * T + t) * hid + m] = w2[r];
    }
    if (tid < hid) b.pb1[pc * hid + tid] = bb;
    else if (tid >= LISA_MAX_HIDDEN && tid - LISA_MAX_HIDDEN < T) b.pb2[pc * T + tid - LISA_MAX_HIDDEN] = bb;
}

// ---------------------------------------------------------------------------
// adaptive weights: the MLP parameters' gradients.  Per (slice, chunk):
//   dW1 += sum_i da_i x_i^T (x_i = [q_i; k_i]), db1 += sum_i da_i,
//   dW2 += sum_i dz_i h_i^T, db2 += sum_i dz_i
// as partial sums; bwd_mlp_reduce adds the partials of every slice and chunk
// in a fixed order.
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_mlp_params(BwdProblem b) {
    constexpr int kTok = 16;
    constexpr int kMaxPer = LISA_MAX_HIDDEN * 2 * D / kThreads;   // dW1 entries per thread
    __shared__ float Xs[kTok][2 * D];
    __shared__ float As[kTok][LISA_MAX_HIDDEN];
    __shared__ float Hs[kTok][LISA_MAX_HIDDEN];
    __shared__ float Zs[kTok][LISA_MAX_T_MLP];
    const Problem &p = b.fwd;
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, tid = threadIdx.x;
    const int T = p.T, hid = p.hidden;
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const size_t sbase = (size_t)sl * p.n * D;
    const TIn *Q = static_cast<const TIn *>(p.Q) + sbase;
    const TIn *K = static_cast<const TIn *>(p.K) + sbase;
    const size_t tb = (size_t)sl * p.n;
    float w1[kMaxPer], w2[2], bb = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxPer; ++r) w1[r] = 0.f;
    w2[0] = w2[1] = 0.f;
    for (int base = t0; base < t1; base += kTok) {
        const int cnt = min(kTok, t1 - base);
        for (int x = tid; x < kTok * 2 * D; x += kThreads) {
            const int j = x / (2 * D), ch = x % (2 * D);
            float v = 0.f;
            if (j < cnt) v = feature(ld((ch < D ? Q : K) + (size_t)(base + j) * D + (ch % D)), p.relu);
            Xs[j][ch] = v;
        }
        for (int x = tid; x < kTok * LISA_MAX_HIDDEN; x += kThreads) {
            const int j = x / LISA_MAX_HIDDEN, m = x % LISA_MAX_HIDDEN;
            const bool in = j < cnt && m < hid;
            As[j][m] = in ? b.dabuf[(tb + base + j) * hid + m] : 0.f;
            Hs[j][m] = in ? b.hbuf[(tb + base + j) * hid + m] : 0.f;
        }
        for (int x = tid; x < kTok * LISA_MAX_T_MLP; x += kThreads) {
            const int j = x / LISA_MAX_T_MLP, t = x % LISA_MAX_T_MLP;
            Zs[j][t] = (j < cnt && t < T) ? b.dzbuf[(tb + base + j) * T + t] : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
#pragma unroll
            for (int r = 0; r < kMaxPer; ++r) {
                const int e = tid + r * kThreads, m = e / (2 * D), ch = e % (2 * D);
                w1[r] = fmaf(As[j][m], Xs[j][ch], w1[r]);
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int e = tid + r * kThreads, t = e / LISA_MAX_HIDDEN, m = e % LISA_MAX_HIDDEN;
                if (t < LISA_MAX_T_MLP) w2[r] = fmaf(Zs[j][t], Hs[j][m], w2[r]);
            }
            if (tid < LISA_MAX_HIDDEN) bb += As[j][tid];
            else if (tid - LISA_MAX_HIDDEN < LISA_MAX_T_MLP) bb += Zs[j][tid - LISA_MAX_HIDDEN];
        }
        __syncthreads();
    }
    const size_t pc = (size_t)sl * p.chunks + c;
#pragma unroll
    for (int r = 0; r < kMaxPer; ++r) {
        const int e = tid + r * kThreads, m = e / (2 * D);
        if (m < hid) b.pw1[pc * hid * 2 * D + e] = w1[r];
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int e = tid + r * kThreads, t = e / LISA_MAX_HIDDEN, m = e % LISA_MAX_HIDDEN;
        if (t < T && m < hid) b.pw2[(pc * T + t) * hid + m] = w2[r];
    }
    if (tid < hid) b.pb1[pc * hid + tid] = bb;
    else if (tid >= LISA_MAX_HIDDEN && tid - LISA_MAX_HIDDEN < T) b.pb2[pc * T + tid - LISA_MAX_HIDDEN] = bb;
}

// 32 consecutive parameter entries per block: warp g sums the partials
// g, g + 8, g + 16, ... of its lane's entry (coalesced 128-byte rows, four
// loads in flight), then lane 0..31 of warp 0 adds the eight warp sums in a
// fixed order.
__global__ void __launch_bounds__(kThreads) bwd_mlp_reduce(BwdProblem b, int D) {
    constexpr int kGroups = kThreads / 32;
    __shared__ float red[kGroups][32];
    const Problem &p = b.fwd;
    const int T = p.T, hid = p.hidden;
    const int n1 = hid * 2 * D, n2 = T * hid;
    const int total = n1 + hid + n2 + T;
    const int parts = p.slices * p.chunks;
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const float *src = nullptr;
    float *dst = nullptr;
    int stride = 0, off = 0;
    if (e < n1) { src = b.pw1; dst = b.dW1; stride = n1; off = e; }
    else if (e < n1 + hid) { src = b.pb1; dst = b.db1; stride = hid; off = e - n1; }
    else if (e < n1 + hid + n2) { src = b.pw2; dst = b.dW2; stride = n2; off = e - n1 - hid; }
    else if (e < total) { src = b.pb2; dst = b.db2; stride = T; off = e - n1 - hid - n2; }
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (src) {
        int r = g;
        for (; r + 3 * kGroups < parts; r += 4 * kGroups) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = src[(size_t)(r + u * kGroups) * stride + off];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] += v[u];
        }
        for (; r < parts; r += kGroups) a[0] += src[(size_t)r * stride + off];
    }
    red[g][lane] = (a[0] + a[1]) + (a[2] + a[3]);
    __syncthreads();
    if (g == 0 && dst) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kGroups; ++k) t += red[k][lane];
        dst[off] = t;
    }
}

// ---------------------------------------------------------------------------
// 6. per slice: ds = sum of the block partials; the slice's dalpha.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) bwd_reduce(BwdProblem b) {
    const int sl = blockIdx.x, tid = threadIdx.x;
    if (tid < D) {   // eight partials in flight per thread, in a fixed order
        const int nds = b.ntile ? b.ntile : b.nblk;   // blocks of the token pass
        b.ds_red[(size_t)sl * D + tid] = sum_partials(b.ds_part + (size_t)sl * nds * D, nds, D, tid);
    }
    if (tid == kThreads - 1) b.dal_slice[sl] = sum_partials(b.dal_part + (size_t)sl * b.nblk, b.nblk, 1, 0);
}

// ---------------------------------------------------------------------------
// 7. dXk = (dK + ds) [Xk > 0], one thread per element; block 0 also writes
// dalpha per head, the sum over the batch in batch order (8.).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_finish_k(BwdProblem b) {
    const Problem &p = b.fwd;
    if (blockIdx.x == 0)
        for (int h = threadIdx.x; h < p.heads; h += kThreads) {
            const int B = p.slices / p.heads;
            float acc = 0.f;
            for (int bb = 0; bb < B; ++bb) acc += b.dal_slice[(size_t)bb * p.heads + h];
            b.dalpha[h] = acc;
        }
    const long long total = (long long)p.slices * p.n * D;
    const TIn *K = static_cast<const TIn *>(p.K);
    TIn *dKo = static_cast<TIn *>(b.dK);
    if constexpr (std::is_same<TIn, __nv_bfloat16>::value) {
        // four channels per thread and step: 16-byte dK loads, 8-byte K loads and stores
        const long long total4 = total / 4;
        for (long long x4 = (long long)blockIdx.x * kThreads + threadIdx.x; x4 < total4;
             x4 += (long long)gridDim.x * kThreads) {
            const long long x = 4 * x4;
            const int ch = (int)(x % D);
            const long long sl = x / ((long long)p.n * D);
            const float4 dk = reinterpret_cast<const float4 *>(b.dk_part)[x4];
            const float4 ds = *reinterpret_cast<const float4 *>(b.ds_red + sl * D + ch);
            const uint2 kb = reinterpret_cast<const uint2 *>(K)[x4];
            const float v[4] = {dk.x + ds.x, dk.y + ds.y, dk.z + ds.z, dk.w + ds.w};
            const float kx[4] = {sm100::bf16_lo(kb.x), sm100::bf16_hi(kb.x), sm100::bf16_lo(kb.y), sm100::bf16_hi(kb.y)};
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = feature_grad(v[e], kx[e], p.relu);
            reinterpret_cast<uint2 *>(dKo)[x4] = make_uint2(sm100::pack_bf16(o[0], o[1]), sm100::pack_bf16(o[2], o[3]));
        }
        return;
    }
    for (long long x = (long long)blockIdx.x * kThreads + threadIdx.x; x < total;
         x += (long long)gridDim.x * kThreads) {
        const int ch = (int)(x % D);
        const long long sl = x / ((long long)p.n * D);
        const float v = b.dk_part[x] + b.ds_red[sl * D + ch];
        st(dKo + x, feature_grad(v, ld(K + x), p.relu));
    }
}

// 4-D map over the window statistics [S][H][W][4] fp32, box {4, 10, 10, 1}.
bool make_map_stats(CUtensorMap *m, const float *lstat, const Problem &p) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {4, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)p.slices};
    cuuint64_t strides[3] = {16, (cuuint64_t)p.W * 16, (cuuint64_t)p.H * p.W * 16};
    cuuint32_t box[4] = {4, (cuuint32_t)kHaloSide, (cuuint32_t)kHaloSide, 1}, es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(lstat), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The backward's second stream, one per device: dUbar's statistics launch
// (fixed weights, tensor-core path) runs there, forked from the caller's
// stream after the key sum and joined back before the reverse recurrence, so
// it overlaps the forward recurrence and the window-statistics pass (they
// share no data).  Created on first use outside stream capture and kept for
// the life of the process; a call made while its stream is being captured
// before that first use runs the launch in line instead.  The mutex also
// keeps concurrent callers' fork ... join sections (which reuse the two
// events) apart.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

SideStream *side_stream(cudaStream_t st) {   // g_side_mu held
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream &ss = g_side[dev];
    if (ss.s) return &ss;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        (void)cudaGetLastError();
        return nullptr;
    }
    cudaStream_t s2 = nullptr;
    cudaEvent_t e1 = nullptr, e2 = nullptr;
    if (cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&e1, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e2, cudaEventDisableTiming) != cudaSuccess) {
        if (e1) cudaEventDestroy(e1);
        if (s2) cudaStreamDestroy(s2);
        (void)cudaGetLastError();
        return nullptr;
    }
    ss.s = s2;
    ss.fork = e1;
    ss.join = e2;
    return &ss;
}

template <typename TIn, int D>
cudaError_t launch_bwd_all(const BwdProblem &b, cudaStream_t st) {
    const Problem &p = b.fwd;
    if (b.tpb != kTpb) return cudaErrorInvalidValue;   // the plan's blocks are kTpb tokens
    cudaError_t err;
    std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
    SideStream *side = nullptr;
    if (!b.mlp && b.tc_dub) {
        side_lock.lock();
        side = side_stream(st);
        if (!side) side_lock.unlock();
    }
    // dUbar / alpha = Q~^T dO: the statistics kernel with dO as its V and K (and the
    // key-sum partials of the first launch)
    auto launch_dub = [&](cudaStream_t s2) {
        Problem q = b.tcfwd;
        q.V = b.dO;
        q.K = b.dO;
        q.k_raw = 1;
        q.tc_part = b.tcdub;
        return launch_tc_stats_partials(q, s2, false);
    };
    if (b.tc_stats) {   // key-sum and [U_1^T ; M^T] partials on the tensor cores
        if ((err = launch_tc_stats_partials(b.tcfwd, st)) != cudaSuccess) return err;
        if (side) {
            if ((err = cudaEventRecord(side->fork, st)) != cudaSuccess ||
                (err = cudaStreamWaitEvent(side->s, side->fork, 0)) != cudaSuccess ||
                (err = launch_dub(side->s)) != cudaSuccess ||
                (err = cudaEventRecord(side->join, side->s)) != cudaSuccess)
                return err;
        }
    } else {
        if ((err = launch_simt(p, st, 0)) != cudaSuccess) return err;   // partial s, K^T V
        if ((err = launch_simt(p, st, 1)) != cudaSuccess) return err;   // partial K^T Q~
    }
    const unsigned grid_stats = (unsigned)p.slices * (unsigned)p.chunks;
    const unsigned grid_tok = (unsigned)p.slices * (unsigned)b.nblk;
    if (D == 64 && b.tc_stats && !p.untruncated)
        bwd_recur_rows<<<(unsigned)p.slices * kRecurSplit, kThreads, 0, st>>>(b);
    else
        bwd_recur<D><<<p.slices, kThreads, 0, st>>>(b);
    if (b.mlp) {   // per-token weights: the MLP's backward, then one dU_k per walk length
        if (std::is_same<TIn, __nv_bfloat16>::value && D == 64 && p.relu != 2) {
            if ((err = cudaFuncSetAttribute(bwd_token_mlp_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kMlpTcSmemBytes)) != cudaSuccess)
                return err;
            bwd_mlp_images<<<(unsigned)(p.slices * b.nh + 1), kThreads, 0, st>>>(b);
            // persistent: two CTAs per SM (its shared memory allows two)
            const unsigned grid_mlp = std::min(grid_tok, 2u * (unsigned)sm_count());
            bwd_token_mlp_tc<<<grid_mlp, kThreads, kMlpTcSmemBytes, st>>>(b);
        } else {
            bwd_token_mlp<TIn, D><<<grid_tok, kThreads, 0, st>>>(b);
        }
        if (p.T > 1) {
            if (std::is_same<TIn, __nv_bfloat16>::value && D == 64 && p.relu != 2)
                bwd_stats_duk_tc<<<dim3(grid_stats, (unsigned)((p.T - 1 + kDukPerBlock - 1) / kDukPerBlock)),
                                   kThreads, 0, st>>>(b);
            else
                bwd_stats_duk<TIn, D><<<dim3(grid_stats, (unsigned)(p.T - 1)), kThreads, 0, st>>>(b);
        }
    } else {
        if (b.tc_dub) {
            if (!side && (err = launch_dub(st)) != cudaSuccess) return err;   // else on the side stream
        } else {
            bwd_stats_dub<TIn, D><<<grid_stats, kThreads, 0, st>>>(b);
        }
        if (std::is_same<TIn, __nv_bfloat16>::value && D == 64 && p.relu != 2)
            bwd_token_a_tc<<<grid_tok, kThreads, 0, st>>>(b);
        else
            bwd_token_a<TIn, D><<<grid_tok, kThreads, 0, st>>>(b);
    }
    if (side) {   // join: the reverse recurrence reads dUbar's partials
        if ((err = cudaStreamWaitEvent(st, side->join, 0)) != cudaSuccess) return err;
        side_lock.unlock();
    }
    if (D == 64 && !p.untruncated && b.tc_dub && p.T <= 3)
        bwd_recur_back_rows<<<(unsigned)p.slices * kRecurSplit, kThreads, 0, st>>>(b);
    else if (D == 64 && !p.untruncated)
        bwd_recur_back_64<<<p.slices, kThreads, 0, st>>>(b);
    else
        bwd_recur_back<D><<<p.slices, kThreads, 0, st>>>(b);
    // bf16 at d = 64 takes the tensor-core token pass, except with the ELU map
    // (its bf16 staging applies ReLU only)
    if (b.ntile) {   // bf16, d = 64, fixed weights: 8 x 8 tiles with their halo in shared memory
        bwd_bimg<<<dim3((unsigned)p.slices, 5), kThreads, 0, st>>>(b);
        auto tile_kern = b.mlp ? bwd_token_b_tile<true> : bwd_token_b_tile<false>;
        if ((err = cudaFuncSetAttribute(tile_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTileSmemBytes)) !=
            cudaSuccess)
            return err;
        // tiled 4-D maps: 10 x 10 halo boxes of the inputs (128-byte swizzle) and of
        // the window statistics ([S][H][W][4] fp32)
        CUtensorMap mK, mV, mQ, mG, mL;
        if (!make_map_grid(&mK, p.K, p.slices, p.H, p.W, kHaloSide, kHaloSide) ||
            !make_map_grid(&mV, p.V, p.slices, p.H, p.W, kHaloSide, kHaloSide) ||
            !make_map_grid(&mQ, p.Q, p.slices, p.H, p.W, kHaloSide, kHaloSide) ||
            !make_map_grid(&mG, b.dO, p.slices, p.H, p.W, kHaloSide, kHaloSide) || !make_map_stats(&mL, b.lstat, p))
            return cudaErrorInvalidValue;
        const long long ntiles = (long long)p.slices * b.ntile;
        const int nsm = sm_count();
        const unsigned grid = (unsigned)(ntiles < nsm ? ntiles : nsm);   // persistent: one CTA per SM
        tile_kern<<<grid, kTileThreads, kTileSmemBytes, st>>>(mK, mV, mQ, mG, mL, b);
    } else {
        constexpr int smem_b = token_b_smem_floats<D>() * (int)sizeof(float);
        if ((err = cudaFuncSetAttribute(bwd_token_b<TIn, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_b)) != cudaSuccess)
            return err;
        bwd_token_b<TIn, D><<<grid_tok, kThreads, smem_b, st>>>(b);
    }
    bwd_reduce<D><<<p.slices, kThreads, 0, st>>>(b);
    const long long total = (long long)p.slices * p.n * D;
    long long blocks = (total + kThreads - 1) / kThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    bwd_finish_k<TIn, D><<<(unsigned)blocks, kThreads, 0, st>>>(b);
    if (b.mlp) {
        if (std::is_same<TIn, __nv_bfloat16>::value && D == 64 && p.relu != 2)
            bwd_mlp_params_tc<<<grid_stats, kThreads, 0, st>>>(b);
        else
            bwd_mlp_params<TIn, D><<<grid_stats, kThreads, 0, st>>>(b);
        const int total = p.hidden * 2 * D + p.hidden + p.T * p.hidden + p.T;
        bwd_mlp_reduce<<<(total + 31) / 32, kThreads, 0, st>>>(b, D);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem &b, cudaStream_t st) {
    const bool bf = (b.fwd.dtype == LISA_BF16);
    switch (b.fwd.D) {
        case 16: return bf ? launch_bwd_all<__nv_bfloat16, 16>(b, st) : launch_bwd_all<float, 16>(b, st);
        case 32: return bf ? launch_bwd_all<__nv_bfloat16, 32>(b, st) : launch_bwd_all<float, 32>(b, st);
        case 64: return bf ? launch_bwd_all<__nv_bfloat16, 64>(b, st) : launch_bwd_all<float, 64>(b, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lisa
