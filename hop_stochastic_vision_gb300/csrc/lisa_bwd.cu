// lisa_bwd.cu -- backward pass of the LiSA layer (fixed walk weights, incl.
// geometric and the untruncated walk): dL/dXq, dL/dXk, dL/dV, dL/dalpha for
// an upstream gradient dO, fp32 arithmetic on CUDA cores, every dtype and
// head width the forward serves.
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
// Launch chain (after the forward's two SIMT statistics kernels, which leave
// the split-K partials of s, U_1 = K^T V and M = K^T Q~):
//   1. bwd_recur      per slice: reduce s, U_1, M; U_k, Ubar (or the solve)
//   2. bwd_stats_dub  per (slice, chunk): partial dUbar = Q~^T (alpha dO)
//   3. bwd_token_a    warp per token: window softmax max / sum, dl_i . l_i,
//                     dalpha terms (per-block partial sums)
//   4. bwd_recur_back per slice: reduce dUbar; G_k; dM, dU_1 (or the solve)
//   5. bwd_token_b    warp per token: dXq, dV, the ds terms (per-block
//                     partial sums) and dK without ds (fp32, workspace)
//   6. bwd_reduce     per slice: ds and the slice's dalpha
//   7. bwd_finish_k   warp per token: dXk = (dK + ds) [Xk > 0]
//   8. bwd_dalpha     dalpha per head = sum over the batch
// Every reduction runs in a fixed order: the result does not depend on
// scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lisa_internal.h"
#include "lisa_solve.cuh"

namespace lisa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float *p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ float relu_if(float x, int relu) { return (relu && x < 0.f) ? 0.f : x; }
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
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
    __syncthreads();
    float *Uk = b.Uk + (size_t)sl * b.nh * D * D;
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
            Uk[idx] = U[idx / D][idx % D];
            ub[x] = p.beta * (1.f - p.beta) * U[idx / D][idx % D];
        }
    } else {
#pragma unroll
        for (int x = 0; x < EPT; ++x) {
            const int idx = tid + x * kThreads;
            Uk[idx] = U[idx / D][idx % D];
            ub[x] = p.T > 1 ? p.w[1] * U[idx / D][idx % D] : 0.f;
        }
        for (int k = 2; k < p.T; ++k) {
            for (int idx = tid; idx < D * D; idx += kThreads) {
                const int a = idx / D, e = idx % D;
                float acc = 0.f;
                for (int c = 0; c < D; ++c) acc = fmaf(M[a][c], U[c][e], acc);
                Un[a][e] = acc;
            }
            __syncthreads();
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const float u = Un[idx / D][idx % D];
                U[idx / D][idx % D] = u;
                Uk[(size_t)(k - 1) * D * D + idx] = u;
                ub[x] = fmaf(p.w[k], u, ub[x]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int x = 0; x < EPT; ++x) b.Ubar[(size_t)sl * D * D + tid + x * kThreads] = ub[x];
}

// ---------------------------------------------------------------------------
// 2. partial dUbar = sum_j Q~_j (alpha dO_j)^T over one chunk.
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_stats_dub(BwdProblem b) {
    constexpr int EPT = D * D / kThreads;
    constexpr int PER_ROW = D / EPT;
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
    const int a = tid / PER_ROW, e0 = (tid % PER_ROW) * EPT;
    float acc[EPT];
#pragma unroll
    for (int x = 0; x < EPT; ++x) acc[x] = 0.f;
    for (int base = t0; base < t1; base += kTile) {
        const int cnt = min(kTile, t1 - base);
        for (int idx = tid; idx < kTile * D; idx += kThreads) {
            const int j = idx / D, ch = idx % D;
            float qv = 0.f, gv = 0.f;
            if (j < cnt) {
                qv = relu_if(ld(Q + (size_t)(base + j) * D + ch), p.relu);
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
            const float qa = Qs[j][a];
#pragma unroll
            for (int x = 0; x < EPT; ++x) acc[x] = fmaf(qa, Gs[j][e0 + x], acc[x]);
        }
        __syncthreads();
    }
    float *out = b.dub_part + ((size_t)sl * p.chunks + c) * D * D;
#pragma unroll
    for (int x = 0; x < EPT; ++x) out[a * D + e0 + x] = acc[x];
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

// Lane l holds channels l and l + 32 (those below D).
template <typename TIn, int D>
__device__ __forceinline__ void load_row(const TIn *row, float (&x)[(D + 31) / 32], int lane, int relu) {
#pragma unroll
    for (int t = 0; t < (D + 31) / 32; ++t) {
        const int ch = lane + 32 * t;
        x[t] = ch < D ? relu_if(ld(row + ch), relu) : 0.f;
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
        // local window
        int nb[9];
        const int cnt = window(i, p.H, p.W, nb);
        float e[9], emax = -INFINITY;
        for (int t9 = 0; t9 < cnt; ++t9) {
            float kr[NC];
            load_row<TIn, D>(K + (size_t)nb[t9] * D, kr, lane, p.relu);
            e[t9] = dot_row<D>(q, kr) * scale;
            emax = fmaxf(emax, e[t9]);
        }
        float l[NC], esum = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) l[t] = 0.f;
        for (int t9 = 0; t9 < cnt; ++t9) {
            const float a = expf(e[t9] - emax);
            esum += a;
            float vr[NC];
            load_row<TIn, D>(V + (size_t)nb[t9] * D, vr, lane, 0);
#pragma unroll
            for (int t = 0; t < NC; ++t) l[t] = fmaf(a, vr[t], l[t]);
        }
        const float inv = 1.f / esum;
        float dgl = 0.f, dll = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            l[t] *= inv;
            dgl = fmaf(go[t], g[t] - l[t], dgl);
            dll = fmaf(go[t], l[t], dll);
        }
        dgl = warp_sum(dgl);
        dll = warp_sum(dll) * (1.f - al);
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
// 4. reduce dUbar; the walk's backward recurrence (or the transposed solve)
// gives dM and dU_1.
// ---------------------------------------------------------------------------
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
        for (int c = 0; c < p.chunks; ++c) acc += b.dub_part[((size_t)sl * p.chunks + c) * D * D + idx];
        dub[x] = acc;
        M[idx / D][idx % D] = b.Mred[(size_t)sl * D * D + idx];
    }
    float *dM = b.dM + (size_t)sl * D * D, *dU1 = b.dU1 + (size_t)sl * D * D;
    const float *Uk = b.Uk + (size_t)sl * b.nh * D * D;
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
            for (int e = 0; e < D; ++e) acc = fmaf(X[e][a], Uk[(size_t)c * D + e], acc);
            dM[idx] = p.beta * acc;
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
            G[idx / D][idx % D] = p.w[p.T - 1] * dub[x];
        }
        __syncthreads();
        for (int k = p.T - 1; k >= 2; --k) {
            // dM += G_k U_(k-1)^T, then G_(k-1) = w_(k-1) dUbar + M^T G_k
            const float *Up = Uk + (size_t)(k - 2) * D * D;
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const int a = idx / D, c = idx % D;
                float acc = 0.f;
                for (int e = 0; e < D; ++e) acc = fmaf(G[a][e], Up[(size_t)c * D + e], acc);
                dm[x] += acc;
            }
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                const int a = idx / D, e = idx % D;
                float acc = p.w[k - 1] * dub[x];
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
        dM[idx] = dm[x];
        dU1[idx] = p.T > 1 ? G[idx / D][idx % D] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// 5. per token j: dXq_j, dV_j, the ds terms -c_j Q_j (per-block sums), and
// dK_j without ds (fp32).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_token_b(BwdProblem b) {
    constexpr int NC = (D + 31) / 32;
    __shared__ float dsw[kWarps][D];
    const Problem &p = b.fwd;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x / b.nblk, blk = blockIdx.x % b.nblk;
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
    const float *Ub = b.Ubar + (size_t)sl * D * D;
    const float *dM = b.dM + (size_t)sl * D * D, *dU1 = b.dU1 + (size_t)sl * D * D;
    const float al = p.alpha[sl % p.heads], w0 = p.w[0];
    const float scale = rsqrtf((float)D);
    float ds[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) ds[t] = 0.f;
    for (int u = warp; u < b.tpb; u += kWarps) {
        const int j = blk * b.tpb + u;
        if (j >= p.n) break;
        float q[NC], k[NC], v[NC], go[NC], sv[NC];
        load_row<TIn, D>(Q + (size_t)j * D, q, lane, p.relu);
        load_row<TIn, D>(K + (size_t)j * D, k, lane, p.relu);
        load_row<TIn, D>(V + (size_t)j * D, v, lane, 0);
        load_row<TIn, D>(dO + (size_t)j * D, go, lane, 0);
#pragma unroll
        for (int t = 0; t < NC; ++t) sv[t] = lane + 32 * t < D ? s[lane + 32 * t] : 0.f;
        const float rq = 1.f / (dot_row<D>(q, sv) + p.eps);
        // dQ~_j[a] = alpha sum_e dO_j[e] Ubar[a][e] + sum_c dM[c][a] K_j[c]
        // dV_j[e]  = w_0 alpha dO_j[e] + sum_a dU_1[a][e] K_j[a]
        // dK_j[a]  = sum_e dU_1[a][e] V_j[e] + sum_c dM[a][c] Q~_j[c]
        float dqt[NC], dv[NC], dk[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            dqt[t] = 0.f;
            dv[t] = w0 * al * go[t];
            dk[t] = 0.f;
        }
        for (int c = 0; c < D; ++c) {
            const float gc = __shfl_sync(0xffffffffu, go[c / 32], c % 32);
            const float kc = __shfl_sync(0xffffffffu, k[c / 32], c % 32);
            const float vc = __shfl_sync(0xffffffffu, v[c / 32], c % 32);
            const float qc = __shfl_sync(0xffffffffu, q[c / 32], c % 32) * rq;
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                const int a = lane + 32 * t;
                if (a < D) {
                    dqt[t] = fmaf(al * gc, Ub[(size_t)a * D + c], dqt[t]);
                    dqt[t] = fmaf(kc, dM[(size_t)c * D + a], dqt[t]);
                    dv[t] = fmaf(kc, dU1[(size_t)c * D + a], dv[t]);
                    dk[t] = fmaf(vc, dU1[(size_t)a * D + c], dk[t]);
                    dk[t] = fmaf(qc, dM[(size_t)a * D + c], dk[t]);
                }
            }
        }
        // through Q~ = Q / r:  c_j = (dQ~_j . Q_j) / r_j^2
        const float cj = dot_row<D>(dqt, q) * rq * rq;
        float dq[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            dq[t] = dqt[t] * rq - cj * sv[t];
            ds[t] = fmaf(-cj, q[t], ds[t]);
        }
        // local window: j as the query (its own softmax row) ...
        int nb[9];
        const int cnt = window(j, p.H, p.W, nb);
        const float4 sj = lst[j];
        const float izj = 1.f / sj.y;
        for (int t9 = 0; t9 < cnt; ++t9) {
            float kr[NC], vr[NC];
            load_row<TIn, D>(K + (size_t)nb[t9] * D, kr, lane, p.relu);
            load_row<TIn, D>(V + (size_t)nb[t9] * D, vr, lane, 0);
            const float a = expf(dot_row<D>(q, kr) * scale - sj.x) * izj;
            const float dlv = dot_row<D>(go, vr) * (1.f - al);
            const float de = a * (dlv - sj.z) * scale;
#pragma unroll
            for (int t = 0; t < NC; ++t) dq[t] = fmaf(de, kr[t], dq[t]);
        }
        // ... and j as a key / value of each neighbour i's row (N is symmetric)
        for (int t9 = 0; t9 < cnt; ++t9) {
            const int i = nb[t9];
            float qi[NC], gi[NC];
            load_row<TIn, D>(Q + (size_t)i * D, qi, lane, p.relu);
            load_row<TIn, D>(dO + (size_t)i * D, gi, lane, 0);
            const float4 si = lst[i];
            const float a = expf(dot_row<D>(qi, k) * scale - si.x) / si.y;
            const float dlv = dot_row<D>(gi, v) * (1.f - al);
            const float de = a * (dlv - si.z) * scale;
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                dv[t] = fmaf(a * (1.f - al), gi[t], dv[t]);
                dk[t] = fmaf(de, qi[t], dk[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            const int ch = lane + 32 * t;
            if (ch < D) {
                const float xq = ld(Q + (size_t)j * D + ch);
                st(dQo + (size_t)j * D + ch, (p.relu && !(xq > 0.f)) ? 0.f : dq[t]);
                st(dVo + (size_t)j * D + ch, dv[t]);
                dKp[(size_t)j * D + ch] = dk[t];
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NC; ++t)
        if (lane + 32 * t < D) dsw[warp][lane + 32 * t] = ds[t];
    __syncthreads();
    for (int ch = threadIdx.x; ch < D; ch += kThreads) {
        float acc = 0.f;
        for (int w = 0; w < kWarps; ++w) acc += dsw[w][ch];
        b.ds_part[((size_t)sl * b.nblk + blk) * D + ch] = acc;
    }
}

// ---------------------------------------------------------------------------
// 6. per slice: ds = sum of the block partials; the slice's dalpha.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) bwd_reduce(BwdProblem b) {
    const int sl = blockIdx.x, tid = threadIdx.x;
    if (tid < D) {
        float acc = 0.f;
        for (int k = 0; k < b.nblk; ++k) acc += b.ds_part[((size_t)sl * b.nblk + k) * D + tid];
        b.ds_red[(size_t)sl * D + tid] = acc;
    }
    if (tid == kThreads - 1) {
        float acc = 0.f;
        for (int k = 0; k < b.nblk; ++k) acc += b.dal_part[(size_t)sl * b.nblk + k];
        b.dal_slice[sl] = acc;
    }
}

// ---------------------------------------------------------------------------
// 7. dXk = (dK + ds) [Xk > 0], one thread per element.
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) bwd_finish_k(BwdProblem b) {
    const Problem &p = b.fwd;
    const long long total = (long long)p.slices * p.n * D;
    const TIn *K = static_cast<const TIn *>(p.K);
    TIn *dKo = static_cast<TIn *>(b.dK);
    for (long long x = (long long)blockIdx.x * kThreads + threadIdx.x; x < total;
         x += (long long)gridDim.x * kThreads) {
        const int ch = (int)(x % D);
        const long long sl = x / ((long long)p.n * D);
        const float v = b.dk_part[x] + b.ds_red[sl * D + ch];
        st(dKo + x, (p.relu && !(ld(K + x) > 0.f)) ? 0.f : v);
    }
}

// ---------------------------------------------------------------------------
// 8. dalpha per head: the sum over the batch, in batch order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) bwd_dalpha(BwdProblem b) {
    const Problem &p = b.fwd;
    const int B = p.slices / p.heads;
    for (int h = blockIdx.x * kThreads + threadIdx.x; h < p.heads; h += gridDim.x * kThreads) {
        float acc = 0.f;
        for (int bb = 0; bb < B; ++bb) acc += b.dal_slice[(size_t)bb * p.heads + h];
        b.dalpha[h] = acc;
    }
}

template <typename TIn, int D>
cudaError_t launch_bwd_all(const BwdProblem &b, cudaStream_t st) {
    const Problem &p = b.fwd;
    cudaError_t err = launch_simt(p, st, 0);   // partial s, K^T V
    if (err != cudaSuccess) return err;
    if ((err = launch_simt(p, st, 1)) != cudaSuccess) return err;   // partial K^T Q~
    const unsigned grid_stats = (unsigned)p.slices * (unsigned)p.chunks;
    const unsigned grid_tok = (unsigned)p.slices * (unsigned)b.nblk;
    bwd_recur<D><<<p.slices, kThreads, 0, st>>>(b);
    bwd_stats_dub<TIn, D><<<grid_stats, kThreads, 0, st>>>(b);
    bwd_token_a<TIn, D><<<grid_tok, kThreads, 0, st>>>(b);
    bwd_recur_back<D><<<p.slices, kThreads, 0, st>>>(b);
    bwd_token_b<TIn, D><<<grid_tok, kThreads, 0, st>>>(b);
    bwd_reduce<D><<<p.slices, kThreads, 0, st>>>(b);
    const long long total = (long long)p.slices * p.n * D;
    long long blocks = (total + kThreads - 1) / kThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    bwd_finish_k<TIn, D><<<(unsigned)blocks, kThreads, 0, st>>>(b);
    bwd_dalpha<<<(p.heads + kThreads - 1) / kThreads, kThreads, 0, st>>>(b);
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
