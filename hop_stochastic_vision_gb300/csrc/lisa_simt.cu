// lisa_simt.cu -- plain SIMT kernel chain of the LiSA forward layer.
//
// Serves every dtype and head width with fp32 arithmetic on CUDA cores: the
// fp32 layer (which stays fp32 end to end) and, as the simple reference
// implementation on the device, the bf16 layer.  Four launches per call:
//
//   1. stats_kv   per (slice, chunk): partial s = sum_j K_j and
//                 partial U_1 = sum_j K_j V_j^T                [note §2.2-2.3]
//   2. stats_kq   per (slice, chunk): s from the partials, Q~_j = Q_j/(Q_j.s+eps),
//                 partial M = sum_j K_j Q~_j^T                 [note §2.3]
//   3. recur      per slice: reduce the partials (fixed chunk order),
//                 U_k = M U_(k-1) for k = 2..T-1, fold sum_k w_k U_k when the
//                 weights are shared by all tokens              [paper Eq. 8]
//   4. epilogue   one warp per token: Q~_i, global term, adaptive weights,
//                 3x3 local branch, alpha mix, store            [note §2.4]
//
// "note" is the reading note of "LiSA: Linear Stochastic Attention for
// Long-Range Visual Modeling" (arXiv 2611.04216v2).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lisa_internal.h"
#include "lisa_solve.cuh"

namespace lisa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;  // tokens staged per step in the stats kernels

__device__ __forceinline__ float load_elem(const float *p) { return *p; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

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

// ---------------------------------------------------------------------------
// 1. partial s and U_1 = K^T V over one chunk of one slice.
// Thread t owns a (D/16) x (D/16) block of U (rows a0.., columns e0..).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) stats_kv_kernel(Problem p) {
    constexpr int RB = D / 16;   // each thread: an RB x RB block of the D x D result
    __shared__ float Ks[kTile][D];
    __shared__ float Vs[kTile][D];
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, tid = threadIdx.x;
    if (blockIdx.x == 0 && tid == 0 && p.err) *p.err = 0;   // first kernel of the chain: clear the error word
    const int t0 = c * p.chunk;
    const int t1 = min(p.n, t0 + p.chunk);
    const TIn *K = static_cast<const TIn *>(p.K) + (size_t)sl * p.n * D;
    const TIn *V = static_cast<const TIn *>(p.V) + (size_t)sl * p.n * D;
    const int a0 = (tid / 16) * RB, e0 = (tid % 16) * RB;
    float acc[RB][RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) acc[r][x] = 0.f;
    float ssum = 0.f;
    for (int base = t0; base < t1; base += kTile) {
        const int cnt = min(kTile, t1 - base);
        for (int idx = tid; idx < kTile * D; idx += kThreads) {
            const int j = idx / D, ch = idx % D;
            float kv = 0.f, vv = 0.f;
            if (j < cnt) {
                kv = feature(load_elem(K + (size_t)(base + j) * D + ch), p.relu);
                vv = load_elem(V + (size_t)(base + j) * D + ch);
            }
            Ks[j][ch] = kv;
            Vs[j][ch] = vv;
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
            float ra[RB], rb[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                ra[r] = Ks[j][a0 + r];
                rb[r] = Vs[j][e0 + r];
            }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int x = 0; x < RB; ++x) acc[r][x] = fmaf(ra[r], rb[x], acc[r][x]);
        }
        if (tid < D)
            for (int j = 0; j < cnt; ++j) ssum += Ks[j][tid];
        __syncthreads();
    }
    const size_t pc = (size_t)sl * p.chunks + c;
    float *U = p.u_part + pc * D * D;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) U[(a0 + r) * D + e0 + x] = acc[r][x];
    if (tid < D) p.s_part[pc * D + tid] = ssum;
}

// ---------------------------------------------------------------------------
// 2. partial M = K^T Q~ over one chunk, Q~_j = Q_j / (Q_j . s + eps).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) stats_kq_kernel(Problem p) {
    constexpr int RB = D / 16;   // each thread: an RB x RB block of the D x D result
    __shared__ float Ks[kTile][D];
    __shared__ float Qs[kTile][D];
    __shared__ float s[D];
    const int c = blockIdx.x % p.chunks, sl = blockIdx.x / p.chunks, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if (tid < D) {
        float acc = 0.f;
        for (int cc = 0; cc < p.chunks; ++cc) acc += p.s_part[((size_t)sl * p.chunks + cc) * D + tid];
        s[tid] = acc;
    }
    __syncthreads();
    const int t0 = c * p.chunk;
    const int t1 = min(p.n, t0 + p.chunk);
    const TIn *Q = static_cast<const TIn *>(p.Q) + (size_t)sl * p.n * D;
    const TIn *K = static_cast<const TIn *>(p.K) + (size_t)sl * p.n * D;
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
            float kv = 0.f, qv = 0.f;
            if (j < cnt) {
                kv = feature(load_elem(K + (size_t)(base + j) * D + ch), p.relu);
                qv = feature(load_elem(Q + (size_t)(base + j) * D + ch), p.relu);
            }
            Ks[j][ch] = kv;
            Qs[j][ch] = qv;
        }
        __syncthreads();
        // row normaliser: one warp per token
        for (int j = warp; j < kTile; j += kThreads / 32) {
            float d = 0.f;
            for (int ch = lane; ch < D; ch += 32) d += Qs[j][ch] * s[ch];
            d = warp_sum(d);
            const float r = 1.f / (d + p.eps);
            __syncwarp();
            for (int ch = lane; ch < D; ch += 32) Qs[j][ch] *= r;
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
            float ra[RB], rb[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                ra[r] = Ks[j][a0 + r];
                rb[r] = Qs[j][e0 + r];
            }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int x = 0; x < RB; ++x) acc[r][x] = fmaf(ra[r], rb[x], acc[r][x]);
        }
        __syncthreads();
    }
    float *M = p.m_part + ((size_t)sl * p.chunks + c) * D * D;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int x = 0; x < RB; ++x) M[(a0 + r) * D + e0 + x] = acc[r][x];
}

// ---------------------------------------------------------------------------
// 3. reduce partials and run the d x d recurrence of one slice.
// Output ucat[slice]: FIXED -> one matrix sum_{k>=1} w_k U_k;
// MLP -> U_1 .. U_(T-1) back to back.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) recur_kernel(Problem p) {
    __shared__ float M[D][D];
    __shared__ float U[D][D];
    __shared__ float Un[D][D];
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
    }
    if (tid < D) {
        float acc = 0.f;
        for (int c = 0; c < p.chunks; ++c) acc += p.s_part[((size_t)sl * p.chunks + c) * D + tid];
        p.s_red[(size_t)sl * D + tid] = acc;
    }
    __syncthreads();
    if (p.untruncated) {
        // U_1 <- (I - beta M)^-1 U_1: A = I - beta M stored transposed in Un, R = U_1
        // transposed in M, the solve's scratch in U (free meanwhile)
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int a = idx / D, b = idx % D;
            Un[b][a] = (a == b ? 1.f : 0.f) - p.beta * M[a][b];
        }
        __syncthreads();
        for (int idx = tid; idx < D * D; idx += kThreads) M[idx % D][idx / D] = U[idx / D][idx % D];
        __syncthreads();
        solve_walk_system<kThreads / 32, (2 * D + kThreads / 32 - 1) / (kThreads / 32)>(&Un[0][0], D, &M[0][0], D, D, D,
                                                                                  &U[0][0], tid);
        for (int idx = tid; idx < D * D; idx += kThreads) U[idx / D][idx % D] = M[idx % D][idx / D];
        __syncthreads();
    }
    const bool folded = (p.wmode != LISA_W_MLP);
    float *out = p.ucat + (size_t)sl * (folded ? 1 : (p.T - 1 > 0 ? p.T - 1 : 1)) * D * D;
    // acc holds sum_k w_k U_k for the entries this thread owns (FIXED mode)
    constexpr int EPT = D * D / kThreads;
    float facc[EPT];
#pragma unroll
    for (int x = 0; x < EPT; ++x) facc[x] = 0.f;
    for (int k = 1; k < p.T; ++k) {
        if (k > 1) {
            for (int idx = tid; idx < D * D; idx += kThreads) {
                const int a = idx / D, e = idx % D;
                float acc = 0.f;
                for (int b = 0; b < D; ++b) acc = fmaf(M[a][b], U[b][e], acc);
                Un[a][e] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < D * D; idx += kThreads) U[idx / D][idx % D] = Un[idx / D][idx % D];
            __syncthreads();
        }
        if (folded) {
#pragma unroll
            for (int x = 0; x < EPT; ++x) {
                const int idx = tid + x * kThreads;
                facc[x] = fmaf(p.w[k], U[idx / D][idx % D], facc[x]);
            }
        } else {
            for (int idx = tid; idx < D * D; idx += kThreads)
                out[(size_t)(k - 1) * D * D + idx] = U[idx / D][idx % D];
        }
    }
    if (folded) {
#pragma unroll
        for (int x = 0; x < EPT; ++x) out[tid + x * kThreads] = facc[x];
    }
}

__device__ __forceinline__ float gelu_erf(float x) {
    return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}

// ---------------------------------------------------------------------------
// 4. epilogue: one warp per token.  Lane l owns channels l, l+32 (< D).
// ---------------------------------------------------------------------------
template <typename TIn, int D>
__global__ void __launch_bounds__(kThreads) epilogue_kernel(Problem p) {
    constexpr int NC = (D + 31) / 32;
    const int lane = threadIdx.x & 31;
    const long long tok = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (tok >= (long long)p.slices * p.n) return;
    const int sl = (int)(tok / p.n), i = (int)(tok % p.n);
    const int r = i / p.W, c = i % p.W;
    const size_t sbase = (size_t)sl * p.n * D;
    const TIn *Q = static_cast<const TIn *>(p.Q) + sbase;
    const TIn *K = static_cast<const TIn *>(p.K) + sbase;
    const TIn *V = static_cast<const TIn *>(p.V) + sbase;
    TIn *O = static_cast<TIn *>(p.O) + sbase;
    const float *s = p.s_red + (size_t)sl * D;

    float q[NC], k[NC], v[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) {
        const int ch = lane + 32 * t;
        q[t] = k[t] = v[t] = 0.f;
        if (ch < D) {
            q[t] = feature(load_elem(Q + (size_t)i * D + ch), p.relu);
            k[t] = feature(load_elem(K + (size_t)i * D + ch), p.relu);
            v[t] = load_elem(V + (size_t)i * D + ch);
        }
    }
    // row normaliser of Q~_i
    float den = 0.f;
#pragma unroll
    for (int t = 0; t < NC; ++t) {
        const int ch = lane + 32 * t;
        if (ch < D) den += q[t] * s[ch];
    }
    const float rq = 1.f / (warp_sum(den) + p.eps);

    // walk weights of this token
    float wk[LISA_MAX_T];
    if (p.wmode == LISA_W_MLP) {
        float z[LISA_MAX_T_MLP];
        for (int t = 0; t < p.T; ++t) z[t] = p.b2[t];
        for (int m = 0; m < p.hidden; ++m) {
            const float *row = p.W1 + (size_t)m * 2 * D;
            float acc = 0.f;
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                const int ch = lane + 32 * t;
                if (ch < D) acc += row[ch] * q[t] + row[D + ch] * k[t];
            }
            const float h = gelu_erf(warp_sum(acc) + p.b1[m]);
            for (int t = 0; t < p.T; ++t) z[t] = fmaf(p.W2[(size_t)t * p.hidden + m], h, z[t]);
        }
        float zmax = z[0];
        for (int t = 1; t < p.T; ++t) zmax = fmaxf(zmax, z[t]);
        float zs = 0.f;
        for (int t = 0; t < p.T; ++t) {
            z[t] = expf(z[t] - zmax);
            zs += z[t];
        }
        for (int t = 0; t < p.T; ++t) wk[t] = z[t] / zs;
    } else {
        for (int t = 0; t < p.T; ++t) wk[t] = p.w[t];
    }

    // global branch g_i = w_0 V_i + sum_{k>=1} w_k Q~_i U_k
    float g[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) g[t] = wk[0] * v[t];
    const int nmat = (p.wmode == LISA_W_MLP) ? p.T - 1 : (p.T > 1 ? 1 : 0);
    const float *Ub = p.ucat + (size_t)sl * (p.wmode == LISA_W_MLP ? (p.T - 1 > 0 ? p.T - 1 : 1) : 1) * D * D;
    for (int mi = 0; mi < nmat; ++mi) {
        const float *Um = Ub + (size_t)mi * D * D;
        float acc[NC];
#pragma unroll
        for (int t = 0; t < NC; ++t) acc[t] = 0.f;
        for (int a = 0; a < D; ++a) {
            const float qa = __shfl_sync(0xffffffffu, q[a / 32], a % 32);
#pragma unroll
            for (int t = 0; t < NC; ++t) {
                const int ch = lane + 32 * t;
                if (ch < D) acc[t] = fmaf(qa, Um[(size_t)a * D + ch], acc[t]);
            }
        }
        const float wm = (p.wmode == LISA_W_MLP) ? wk[mi + 1] : 1.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) g[t] = fmaf(wm * rq, acc[t], g[t]);
    }

    // local 3x3 branch over in-grid neighbours
    const float scale = rsqrtf((float)D);
    float e[9];
    int nb[9];
    int cnt = 0;
    for (int dr = -1; dr <= 1; ++dr)
        for (int dc = -1; dc <= 1; ++dc) {
            const int rr = r + dr, cc = c + dc;
            if (rr < 0 || rr >= p.H || cc < 0 || cc >= p.W) continue;
            nb[cnt++] = rr * p.W + cc;
        }
    float emax = -INFINITY;
    for (int t9 = 0; t9 < cnt; ++t9) {
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            const int ch = lane + 32 * t;
            if (ch < D) acc += q[t] * feature(load_elem(K + (size_t)nb[t9] * D + ch), p.relu);
        }
        e[t9] = warp_sum(acc) * scale;
        emax = fmaxf(emax, e[t9]);
    }
    float l[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) l[t] = 0.f;
    float esum = 0.f;
    for (int t9 = 0; t9 < cnt; ++t9) {
        const float a = expf(e[t9] - emax);
        esum += a;
#pragma unroll
        for (int t = 0; t < NC; ++t) {
            const int ch = lane + 32 * t;
            if (ch < D) l[t] = fmaf(a, load_elem(V + (size_t)nb[t9] * D + ch), l[t]);
        }
    }
    const float inv = 1.f / esum;
    const float al = p.alpha[sl % p.heads];
#pragma unroll
    for (int t = 0; t < NC; ++t) {
        const int ch = lane + 32 * t;
        if (ch < D) store_elem(O + (size_t)i * D + ch, al * g[t] + (1.f - al) * (l[t] * inv));
    }
}

template <typename TIn, int D>
cudaError_t launch_all(const Problem &p, cudaStream_t st, int stage) {
    const unsigned grid_stats = (unsigned)p.slices * (unsigned)p.chunks;
    if (stage < 0 || stage == 0) stats_kv_kernel<TIn, D><<<grid_stats, kThreads, 0, st>>>(p);
    if (stage < 0 || stage == 1) stats_kq_kernel<TIn, D><<<grid_stats, kThreads, 0, st>>>(p);
    if (stage < 0 || stage == 2) recur_kernel<D><<<p.slices, kThreads, 0, st>>>(p);
    if (stage < 0 || stage == 3) {
        const long long toks = (long long)p.slices * p.n;
        const long long blocks = (toks + kThreads / 32 - 1) / (kThreads / 32);
        epilogue_kernel<TIn, D><<<(unsigned)blocks, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

const char *const kSimtStageNames[kSimtStages] = {"stats_kv", "stats_kq", "recur", "epilogue"};

cudaError_t launch_simt(const Problem &p, cudaStream_t st, int stage) {
    const bool bf = (p.dtype == LISA_BF16);
    switch (p.D) {
        case 16: return bf ? launch_all<__nv_bfloat16, 16>(p, st, stage) : launch_all<float, 16>(p, st, stage);
        case 32: return bf ? launch_all<__nv_bfloat16, 32>(p, st, stage) : launch_all<float, 32>(p, st, stage);
        case 64: return bf ? launch_all<__nv_bfloat16, 64>(p, st, stage) : launch_all<float, 64>(p, st, stage);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lisa
