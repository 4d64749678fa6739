// lisa_tc.cu -- tensor-core kernel chain of the LiSA forward layer for bf16
// layers with d_h = d_v = 64 on sm_103a.
//
// "note" below is the reading note of "LiSA: Linear Stochastic Attention for
// Long-Range Visual Modeling" (arXiv 2611.04216v2).  Four launches, chained
// with programmatic dependent launch so each kernel's prologue (TMEM
// allocation, barrier set-up, TMA prefetch of its own inputs) overlaps the
// previous kernel's tail:
//
//   1. keysum   s = sum_j K_j, split over token chunks           [note §2.2]
//   2. stats    per chunk, one tcgen05 MMA chain over the tokens:
//                 [V | Q~]^T K = [U_1^T ; M^T]   (128 x 64, fp32 in TMEM)
//               with Q~_j = Q_j / (Q_j . s + eps) formed in shared memory;
//               the chunks of a thread-block cluster sum their results in
//               distributed shared memory (fixed order)        [note §2.3]
//   3. recur    per slice: U_k^T = U_(k-1)^T M^T, fold sum_k w_k U_k^T
//               (or keep U_1..U_(T-1) for per-token weights), and emit the
//               epilogue's B operand [U^T rows | s_hi | s_lo] in bf16  [Eq. 8]
//   4. epilogue per 128-token tile of the grid:
//               tcgen05: Q [U | s] -> Q U and Q . s (so Q~ U = (Q U)/(Q.s+eps))
//               and, with adaptive weights, [Q | K] W1^T for the MLP;
//               mma.sync: the 3x3 local branch on 4x4-token blocks (scores
//               against the 6x6 key window, masked softmax, weights times V);
//               then alpha mix and a TMA store                    [note §2.4]
//
// Shared-memory operands use the 128-byte swizzle that TMA writes: one token
// row of 64 bf16 is 128 bytes, 8 rows form a 1024-byte atom.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "lisa_internal.h"
#include "lisa_sm100.cuh"

namespace lisa {
namespace {

using namespace sm100;

constexpr int kD = 64;             // head width of this family
constexpr int kRow = 128;          // bytes of one token row (64 bf16)
constexpr int kSub = 64;           // tokens per stats pipeline stage
constexpr int kStages = 3;         // stats pipeline depth
constexpr int kStageBytes = 3 * kSub * kRow;   // V | Q~ | K
constexpr int kRecurRowBlocks = 4; // recur CTAs per slice (16 rows of U^T each)
constexpr int kRedStride = 68;     // fp32 row stride of the cluster-reduction buffer
constexpr int kXStride = 68;       // fp32 row stride of the epilogue exchange buffer

// error word bits
constexpr int kErrTimeoutLoad = 1;
constexpr int kErrTimeoutMma = 2;

struct TcParams {
    int slices, heads, H, W, n, T, relu, wmode, hidden;
    float eps;
    const float *alpha;
    float w[LISA_MAX_T];
    const float *W1, *b1, *W2, *b2;
    const void *K;
    int chunks, chunk, cl, parts;    // split-K plan; cluster size; partials per slice
    int th, tw, tiles_r, tiles_c;    // epilogue tile (th x tw = 128 tokens)
    int n_umat, epi_rows, n_mlp;     // epilogue B operand: U blocks, rows, MLP width (x16)
    float *s_part;                   // [S][C][64]
    float *part;                     // [S][P][128][64]
    uint8_t *bepi;                   // [S][epi_rows][128] bf16, 128-B swizzled rows
    uint8_t *w1img;                  // [2][n_mlp][128] bf16 (W1 q-part | k-part), swizzled
    int *err;
};

__device__ __forceinline__ void record_error(int *err, int bits) { atomicOr(err, bits); }

__device__ __forceinline__ uint32_t relu2(uint32_t v) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&v);
    __nv_bfloat162 z = __float2bfloat162_rn(0.f);
    x = __hmax2(x, z);
    return *reinterpret_cast<uint32_t *>(&x);
}
__device__ __forceinline__ uint4 relu4(uint4 v) {
    return make_uint4(relu2(v.x), relu2(v.y), relu2(v.z), relu2(v.w));
}
// In-place ReLU of `bytes` (multiple of 16) of shared memory.
__device__ __forceinline__ void relu_smem(uint8_t *p, int bytes, int tid, int nthreads) {
    uint4 *v = reinterpret_cast<uint4 *>(p);
    for (int i = tid; i < bytes / 16; i += nthreads) v[i] = relu4(v[i]);
}

// ===========================================================================
// 1. keysum: partial s over a chunk of tokens (ReLU applied), fp32.
// ===========================================================================
__global__ void __launch_bounds__(256) tc_keysum_kernel(TcParams p) {
    __shared__ float red[32][kD + 1];
    const int sl = blockIdx.x / p.chunks, c = blockIdx.x % p.chunks;
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.err = 0;
    pdl_launch_dependents();
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const int cg = threadIdx.x & 7, j0 = threadIdx.x >> 3;
    const uint4 *K = static_cast<const uint4 *>(p.K) + (size_t)sl * p.n * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    int j = t0 + j0;
    for (; j + 96 < t1; j += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(K + (size_t)(j + 32 * u) * 8 + cg);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 x = p.relu ? relu4(v[u]) : v[u];
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += bf16_lo(w4[e]);
                acc[2 * e + 1] += bf16_hi(w4[e]);
            }
        }
    }
    for (; j < t1; j += 32) {
        uint4 x = __ldg(K + (size_t)j * 8 + cg);
        if (p.relu) x = relu4(x);
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[2 * e] += bf16_lo(w4[e]);
            acc[2 * e + 1] += bf16_hi(w4[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[j0][cg * 8 + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < kD) {
        float s = 0.f;
        for (int r = 0; r < 32; ++r) s += red[r][threadIdx.x];
        p.s_part[((size_t)sl * p.chunks + c) * kD + threadIdx.x] = s;
    }
}

// ===========================================================================
// 2. stats: [U_1^T ; M^T] of a chunk on tcgen05, cluster-reduced.
// ===========================================================================
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void stats_issue_loads(const CUtensorMap *mQ, const CUtensorMap *mK,
                                                  const CUtensorMap *mV, uint32_t stage_base,
                                                  uint32_t bar, int tok, int sl) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(stage_base, mV, 0, tok, sl, bar);
    tma_load_3d(stage_base + kSub * kRow, mQ, 0, tok, sl, bar);
    tma_load_3d(stage_base + 2 * kSub * kRow, mK, 0, tok, sl, bar);
}

__global__ void __launch_bounds__(128) tc_stats_kernel(const __grid_constant__ CUtensorMap mQ,
                                                       const __grid_constant__ CUtensorMap mK,
                                                       const __grid_constant__ CUtensorMap mV,
                                                       TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], done_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ float s_sh[kD];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sl = blockIdx.x / p.chunks, c = blockIdx.x % p.chunks;
    const int t0 = c * p.chunk;
    const int ntok = max(0, min(p.n, t0 + p.chunk) - t0);
    const int nsub = (ntok + kSub - 1) / kSub;
    const uint32_t base = smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    // Inputs do not depend on the previous kernel: start streaming them now.
    if (tid == 0)
        for (int i = 0; i < kStages && i < nsub; ++i)
            stats_issue_loads(&mQ, &mK, &mV, base + i * kStageBytes, smem_u32(&full_bar[i]),
                              t0 + i * kSub, sl);
    pdl_wait();  // s partials are complete
    if (tid < kD) {
        float s = 0.f;
        for (int cc = 0; cc < p.chunks; ++cc) s += p.s_part[((size_t)sl * p.chunks + cc) * kD + tid];
        s_sh[tid] = s;
    }
    __syncthreads();

    constexpr uint32_t idesc = make_idesc_bf16(128, 64, true, true);
    bool ok = true;
    for (int i = 0; i < nsub; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(smem_u32(&full_bar[st]), ph)) {
            record_error(p.err, kErrTimeoutLoad);
            ok = false;
        }
        if (!__syncthreads_and(ok)) break;
        uint8_t *Vb = sm + st * kStageBytes;
        uint8_t *Qb = Vb + kSub * kRow;
        uint8_t *Kb = Qb + kSub * kRow;
        if (p.relu) relu_smem(Kb, kSub * kRow, tid, 128);
        {   // Q~_j = Q_j / (Q_j . s + eps): two threads per token, 32 features each
            const int j = tid >> 1, h = tid & 1;
            uint4 q[4];
            float dot = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int chunk = 4 * h + k;
                q[k] = *reinterpret_cast<uint4 *>(Qb + sw128_offset(j, chunk));
                if (p.relu) q[k] = relu4(q[k]);
                const uint32_t w4[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dot = fmaf(bf16_lo(w4[e]), s_sh[chunk * 8 + 2 * e], dot);
                    dot = fmaf(bf16_hi(w4[e]), s_sh[chunk * 8 + 2 * e + 1], dot);
                }
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            const float r = 1.f / (dot + p.eps);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t w4[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
                uint4 o;
                o.x = pack_bf16(bf16_lo(w4[0]) * r, bf16_hi(w4[0]) * r);
                o.y = pack_bf16(bf16_lo(w4[1]) * r, bf16_hi(w4[1]) * r);
                o.z = pack_bf16(bf16_lo(w4[2]) * r, bf16_hi(w4[2]) * r);
                o.w = pack_bf16(bf16_lo(w4[3]) * r, bf16_hi(w4[3]) * r);
                *reinterpret_cast<uint4 *>(Qb + sw128_offset(j, 4 * h + k)) = o;
            }
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t vaddr = base + st * kStageBytes;
            const uint32_t kaddr = vaddr + 2 * kSub * kRow;
#pragma unroll
            for (int ks = 0; ks < kSub / 16; ++ks) {
                const uint64_t ad = make_desc_sw128(vaddr + ks * 2048, kSub * kRow, 1024);
                const uint64_t bd = make_desc_sw128(kaddr + ks * 2048, 1024, 1024);
                tc_mma(tmem, ad, bd, idesc, (i | ks) != 0);
            }
            tc_commit(smem_u32(&empty_bar[st]));
            // refill the stage the previous sub-chunk used
            const int prev = i - 1, nxt = prev + kStages;
            if (prev >= 0 && nxt < nsub) {
                const int pst = prev % kStages;
                if (!mbar_wait(smem_u32(&empty_bar[pst]), (prev / kStages) & 1)) {
                    record_error(p.err, kErrTimeoutMma);
                } else {
                    stats_issue_loads(&mQ, &mK, &mV, base + pst * kStageBytes,
                                      smem_u32(&full_bar[pst]), t0 + nxt * kSub, sl);
                }
            }
        }
    }
    if (tid == 0) tc_commit(smem_u32(&done_bar));
    if (!mbar_wait(smem_u32(&done_bar), 0)) record_error(p.err, kErrTimeoutMma);
    tc_fence_after();

    // TMEM -> shared: thread owns row 32*warp + lane of the 128 x 64 result
    float *red = reinterpret_cast<float *>(sm);
    const int row = 32 * warp + lane;
#pragma unroll
    for (int cb = 0; cb < 64; cb += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + cb, r);
        tc_wait_ld();
        float4 *dst = reinterpret_cast<float4 *>(red + row * kRedStride + cb);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                 __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
    }
    tc_fence_before();
    cluster_sync();

    // rank q of the cluster sums rows q, q + CL, ... over the cluster's CTAs
    const uint32_t rank = cluster_rank();
    const int CL = p.cl;
    const int pidx = c / CL;
    float *out = p.part + ((size_t)sl * p.parts + pidx) * 128 * kD;
    const int my_rows = (128 - (int)rank + CL - 1) / CL;
    const uint32_t red_base = smem_u32(red);
    for (int item = tid; item < my_rows * 16; item += 128) {
        const int rr = (int)rank + CL * (item >> 4);
        const int f = item & 15;
        const uint32_t off = (uint32_t)(rr * kRedStride + 4 * f) * 4u;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int qq = 0; qq < CL; ++qq) {
            const float4 v = ld_dsmem4(map_rank(red_base + off, (uint32_t)qq));
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4 *>(out + rr * kD)[f] = acc;
    }
    cluster_sync();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ===========================================================================
// 3. recur: partial reduction, U_k^T = U_(k-1)^T M^T, epilogue operand.
// ===========================================================================
// Writes one 64-element fp32 row as bf16 into a 128-B-swizzled row image.
__device__ __forceinline__ void put_row_bf16(uint8_t *img, int row, const float *v, int chunk) {
    uint4 o;
    o.x = pack_bf16(v[0], v[1]);
    o.y = pack_bf16(v[2], v[3]);
    o.z = pack_bf16(v[4], v[5]);
    o.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(img + (size_t)row * kRow + ((chunk ^ (row & 7)) << 4)) = o;
}

__global__ void __launch_bounds__(256) tc_recur_kernel(TcParams p) {
    __shared__ float Mt[kD][kD + 1];     // M^T [b][a]
    __shared__ float Ut[16][kD + 1];     // this CTA's 16 rows of U_k^T
    __shared__ float Un[16][kD + 1];
    __shared__ float Fold[16][kD + 1];
    const int tid = threadIdx.x;
    const int sl = blockIdx.x / kRecurRowBlocks, rb = blockIdx.x % kRecurRowBlocks;
    pdl_launch_dependents();
    pdl_wait();
    const float *part = p.part + (size_t)sl * p.parts * 128 * kD;
    for (int idx = tid; idx < kD * kD; idx += 256) {
        const int b = idx / kD, a = idx % kD;
        float m = 0.f;
        for (int q = 0; q < p.parts; ++q) m += part[((size_t)q * 128 + kD + b) * kD + a];
        Mt[b][a] = m;
    }
    for (int idx = tid; idx < 16 * kD; idx += 256) {
        const int e = idx / kD, a = idx % kD;
        float u = 0.f;
        for (int q = 0; q < p.parts; ++q) u += part[((size_t)q * 128 + 16 * rb + e) * kD + a];
        Ut[e][a] = u;
        Fold[e][a] = 0.f;
    }
    __syncthreads();
    const bool folded = (p.wmode != LISA_W_MLP);
    uint8_t *img = p.bepi + (size_t)sl * p.epi_rows * kRow;
    for (int k = 1; k < p.T; ++k) {
        if (k > 1) {
            for (int idx = tid; idx < 16 * kD; idx += 256) {
                const int e = idx / kD, a = idx % kD;
                float acc = 0.f;
#pragma unroll 8
                for (int b = 0; b < kD; ++b) acc = fmaf(Ut[e][b], Mt[b][a], acc);
                Un[e][a] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < 16 * kD; idx += 256) Ut[idx / kD][idx % kD] = Un[idx / kD][idx % kD];
            __syncthreads();
        }
        if (folded) {
            for (int idx = tid; idx < 16 * kD; idx += 256)
                Fold[idx / kD][idx % kD] = fmaf(p.w[k], Ut[idx / kD][idx % kD], Fold[idx / kD][idx % kD]);
        } else if (tid < 128) {
            const int e = tid >> 3, chunk = tid & 7;
            put_row_bf16(img, (k - 1) * kD + 16 * rb + e, &Ut[e][chunk * 8], chunk);
        }
        __syncthreads();
    }
    if (folded && tid < 128) {
        const int e = tid >> 3, chunk = tid & 7;
        put_row_bf16(img, 16 * rb + e, &Fold[e][chunk * 8], chunk);
    }
    if (rb == 0 && tid < 128) {
        // rows n_umat*64 + {0: s_hi, 1: s_lo, 2..15: 0}
        __shared__ float srow[2][kD];
        if (tid < kD) {
            float s = 0.f;
            for (int cc = 0; cc < p.chunks; ++cc) s += p.s_part[((size_t)sl * p.chunks + cc) * kD + tid];
            const float hi = __bfloat162float(__float2bfloat16_rn(s));
            srow[0][tid] = hi;
            srow[1][tid] = s - hi;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int r16 = tid >> 3, chunk = tid & 7;
        float zero[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float *src = r16 < 2 ? &srow[r16][chunk * 8] : zero;
        put_row_bf16(img, p.n_umat * kD + r16, src, chunk);
    }
    if (!folded && sl == 0 && rb == 0) {
        // W1 [hidden][2*64] -> two K-major images [n_mlp rows][64]: q-part, k-part
        for (int idx = tid; idx < 2 * p.n_mlp * 8; idx += 256) {
            const int half = idx / (p.n_mlp * 8), rem = idx % (p.n_mlp * 8);
            const int m = rem >> 3, chunk = rem & 7;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = m < p.hidden ? p.W1[(size_t)m * 2 * kD + half * kD + chunk * 8 + e] : 0.f;
            put_row_bf16(p.w1img + (size_t)half * p.n_mlp * kRow, m, v, chunk);
        }
    }
}

// ===========================================================================
// 4. epilogue
// ===========================================================================
struct EpiLayout {
    uint32_t q, kh, vh, bepi, kt, w1, x, total;
};

__host__ __device__ inline uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

__host__ __device__ inline EpiLayout epi_layout(int th, int tw, int epi_rows, int n_mlp, bool mlp) {
    EpiLayout L;
    const uint32_t halo = align1k((uint32_t)(th + 2) * (tw + 2) * kRow);
    uint32_t off = 0;
    L.q = off; off += 128 * kRow;
    L.kh = off; off += halo;
    L.vh = off; off += halo;
    L.bepi = off; off += align1k((uint32_t)epi_rows * kRow);
    L.kt = off; if (mlp) off += 128 * kRow;
    L.w1 = off; if (mlp) off += align1k(2u * n_mlp * kRow);
    L.x = off; off += 128u * kXStride * 4u;
    L.total = off;
    return L;
}

__device__ __forceinline__ float gelu_erf(float x) {
    return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}

__global__ void __launch_bounds__(256) tc_epilogue_kernel(const __grid_constant__ CUtensorMap mQ,
                                                          const __grid_constant__ CUtensorMap mKh,
                                                          const __grid_constant__ CUtensorMap mVh,
                                                          const __grid_constant__ CUtensorMap mKt,
                                                          const __grid_constant__ CUtensorMap mO,
                                                          TcParams p, uint32_t tmem_cols) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t load_bar, bepi_bar, mma_bar;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool mlp = (p.wmode == LISA_W_MLP);
    const int th = p.th, tw = p.tw, hw = tw + 2;
    const EpiLayout L = epi_layout(th, tw, p.epi_rows, p.n_mlp, mlp);
    const int tiles = p.tiles_r * p.tiles_c;
    const int sl = blockIdx.x / tiles, tix = blockIdx.x % tiles;
    const int r0 = (tix / p.tiles_c) * th, c0 = (tix % p.tiles_c) * tw;
    const uint32_t base = smem_u32(sm);
    const uint32_t halo_rows = (uint32_t)(th + 2) * hw;

    if (tid == 0) {
        mbar_init(smem_u32(&load_bar), 1);
        mbar_init(smem_u32(&bepi_bar), 1);
        mbar_init(smem_u32(&mma_bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    if (tid == 0) {  // this tile's inputs: independent of the earlier kernels
        const uint32_t bytes = (128u + 2u * halo_rows + (mlp ? 128u : 0u)) * kRow;
        const uint32_t lb = smem_u32(&load_bar);
        mbar_arrive_expect_tx(lb, bytes);
        tma_load_4d(base + L.q, &mQ, 0, c0, r0, sl, lb);
        tma_load_4d(base + L.kh, &mKh, 0, c0 - 1, r0 - 1, sl, lb);
        tma_load_4d(base + L.vh, &mVh, 0, c0 - 1, r0 - 1, sl, lb);
        if (mlp) tma_load_4d(base + L.kt, &mKt, 0, c0, r0, sl, lb);
    }
    pdl_wait();  // the B operand of this slice is ready
    if (tid == 0) {
        const uint32_t bb = smem_u32(&bepi_bar);
        const uint32_t bbytes = (uint32_t)p.epi_rows * kRow;
        const uint32_t wbytes = mlp ? 2u * p.n_mlp * kRow : 0u;
        mbar_arrive_expect_tx(bb, bbytes + wbytes);
        bulk_load(base + L.bepi, p.bepi + (size_t)sl * p.epi_rows * kRow, bbytes, bb);
        if (mlp) bulk_load(base + L.w1, p.w1img, wbytes, bb);
    }
    bool ok = mbar_wait(smem_u32(&load_bar), 0);
    if (!ok) record_error(p.err, kErrTimeoutLoad);
    if (p.relu) {
        relu_smem(sm + L.q, 128 * kRow, tid, 256);
        relu_smem(sm + L.kh, (int)halo_rows * kRow, tid, 256);
        if (mlp) relu_smem(sm + L.kt, 128 * kRow, tid, 256);
    }
    fence_proxy_async();
    __syncthreads();

    // ---- tensor-core products (one thread issues, completion on mma_bar)
    if (tid == 0) {
        if (!mbar_wait(smem_u32(&bepi_bar), 0)) record_error(p.err, kErrTimeoutLoad);
        tc_fence_after();
        for (int r = 0; r < p.epi_rows; r += 256) {
            const int N = min(256, p.epi_rows - r);
            const uint32_t idesc = make_idesc_bf16(128, N, false, false);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = make_desc_sw128(base + L.q + ks * 32, 16, 1024);
                const uint64_t bd = make_desc_sw128(base + L.bepi + r * kRow + ks * 32, 16, 1024);
                tc_mma(tmem + r, ad, bd, idesc, ks > 0);
            }
        }
        if (mlp) {
            const uint32_t idesc = make_idesc_bf16(128, p.n_mlp, false, false);
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t abase = (ks < 4 ? L.q : L.kt) + (ks & 3) * 32;
                const uint32_t bbase = L.w1 + (ks < 4 ? 0u : (uint32_t)p.n_mlp * kRow) + (ks & 3) * 32;
                tc_mma(tmem + p.epi_rows, make_desc_sw128(base + abase, 16, 1024),
                       make_desc_sw128(base + bbase, 16, 1024), idesc, ks > 0);
            }
        }
        tc_commit(smem_u32(&mma_bar));
    }

    // ---- 3x3 local branch on the legacy tensor path: warp w owns 4x4 block w
    const int g = lane >> 2, q4 = lane & 3;
    const int bpr = tw >> 2;
    const int bi = warp / bpr, bj = warp % bpr;
    float lacc[8][4];
    {
        // A fragments: the block's 16 query rows, 4 k-steps of 16 channels
        uint32_t a[4][4];
        {
            const int ml = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int trow = (4 * bi + (ml >> 2)) * tw + 4 * bj + (ml & 3);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(base + L.q + sw128_offset(trow, 2 * ks + (lane >> 4)), a[ks][0], a[ks][1],
                        a[ks][2], a[ks][3]);
        }
        // window key kappa (0..35) -> halo row; padding keys point at key 0
        auto halo_row = [&](int kappa) -> uint32_t {
            if (kappa >= 36) kappa = 0;
            return (uint32_t)((4 * bi + kappa / 6) * hw + 4 * bj + kappa % 6);
        };
        float sc[5][4];
#pragma unroll
        for (int j = 0; j < 5; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
                const int kappa = 8 * (2 * pr + (lane >> 4)) + (lane & 7);
                const int chunk = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(base + L.kh + sw128_offset(halo_row(kappa), chunk), b0, b1, b2, b3);
                mma_bf16_16816(sc[2 * pr], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
                if (pr < 2) mma_bf16_16816(sc[2 * pr + 1], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b2, b3);
            }
        }
        // mask: key in the 3x3 window of the query and inside the grid
        const float c2 = 1.4426950408889634f * 0.125f;   // log2(e) / sqrt(64)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 5; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = g + 8 * (e >> 1);
                const int kappa = 8 * j + 2 * q4 + (e & 1);
                const int ka = kappa / 6, kb = kappa % 6;
                const int du = ka - (m >> 2), dv = kb - (m & 3);
                const int gr = r0 + 4 * bi + ka - 1, gc = c0 + 4 * bj + kb - 1;
                const bool valid = kappa < 36 && du >= 0 && du <= 2 && dv >= 0 && dv <= 2 &&
                                   gr >= 0 && gr < p.H && gc >= 0 && gc < p.W;
                sc[j][e] = valid ? sc[j][e] * c2 : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], sc[j][e]);
            }
        float sum[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            if (mx[h] == -INFINITY) mx[h] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 5; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sc[j][e] = exp2f(sc[j][e] - mx[e >> 1]);
                sum[e >> 1] += sc[j][e];
            }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
            sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
        }
        const float inv[2] = {sum[0] > 0.f ? 1.f / sum[0] : 0.f, sum[1] > 0.f ? 1.f / sum[1] : 0.f};
        // weights as A fragments (keys are the k dimension), times V window
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) lacc[nt][0] = lacc[nt][1] = lacc[nt][2] = lacc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 3; ++ks) {
            const int j0 = 2 * ks, j1 = 2 * ks + 1;
            const uint32_t pa0 = pack_bf16(sc[j0][0], sc[j0][1]);
            const uint32_t pa1 = pack_bf16(sc[j0][2], sc[j0][3]);
            const uint32_t pa2 = j1 < 5 ? pack_bf16(sc[j1][0], sc[j1][1]) : 0u;
            const uint32_t pa3 = j1 < 5 ? pack_bf16(sc[j1][2], sc[j1][3]) : 0u;
            const int kappa = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
            const uint32_t hrow = halo_row(kappa);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(base + L.vh + sw128_offset(hrow, 2 * np + (lane >> 4)), b0, b1, b2, b3);
                mma_bf16_16816(lacc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
                mma_bf16_16816(lacc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            lacc[nt][0] *= inv[0]; lacc[nt][1] *= inv[0];
            lacc[nt][2] *= inv[1]; lacc[nt][3] *= inv[1];
        }
    }

    // ---- global branch from TMEM: thread = tile row, half the channels
    const float alpha = p.alpha[sl % p.heads];
    float *X = reinterpret_cast<float *>(sm + L.x);
    if (!mbar_wait(smem_u32(&mma_bar), 0)) record_error(p.err, kErrTimeoutMma);
    tc_fence_after();
    {
        const int quad = warp & 3, half = warp >> 2;
        const int row = 32 * quad + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
        uint32_t r[16];
        tmem_ld16(tl + p.n_umat * kD, r);   // Q.s_hi, Q.s_lo
        tc_wait_ld();
        const float rq = 1.f / (__uint_as_float(r[0]) + __uint_as_float(r[1]) + p.eps);
        float wk[LISA_MAX_T];
        if (mlp) {
            float z[LISA_MAX_T_MLP];
            for (int t = 0; t < p.T; ++t) z[t] = p.b2[t];
            for (int cb = 0; cb < p.n_mlp; cb += 16) {
                tmem_ld16(tl + p.epi_rows + cb, r);
                tc_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int m = cb + k;
                    if (m < p.hidden) {
                        const float hv = gelu_erf(__uint_as_float(r[k]) + p.b1[m]);
                        for (int t = 0; t < p.T; ++t) z[t] = fmaf(p.W2[t * p.hidden + m], hv, z[t]);
                    }
                }
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
            wk[0] = p.w[0];
        }
        float acc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] = 0.f;
        for (int u = 0; u < p.n_umat; ++u) {
            const float wu = mlp ? wk[u + 1] : 1.f;
#pragma unroll
            for (int cb = 0; cb < 32; cb += 16) {
                tmem_ld16(tl + u * kD + 32 * half + cb, r);
                tc_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) acc[cb + k] = fmaf(wu, __uint_as_float(r[k]), acc[cb + k]);
            }
        }
        // V_i (row `row` of the tile) from the halo buffer
        const int tr = row / tw, tcl = row % tw;
        const int hrow = (tr + 1) * hw + tcl + 1;
        float *xr = X + row * kXStride + 32 * half;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int chunk = 4 * half + k;
            const uint4 v = *reinterpret_cast<const uint4 *>(sm + L.vh + sw128_offset(hrow, chunk));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            float o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[2 * e] = alpha * (wk[0] * bf16_lo(w4[e]) + rq * acc[8 * k + 2 * e]);
                o[2 * e + 1] = alpha * (wk[0] * bf16_hi(w4[e]) + rq * acc[8 * k + 2 * e + 1]);
            }
            reinterpret_cast<float4 *>(xr + 8 * k)[0] = make_float4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<float4 *>(xr + 8 * k)[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- mix and store: warp w writes its 4x4 block into the output tile
    {
        const float beta_l = 1.f - alpha;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = g + 8 * h;
            const int trow = (4 * bi + (m >> 2)) * tw + 4 * bj + (m & 3);
            const float *xr = X + trow * kXStride;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int ch = 8 * nt + 2 * q4;
                const float2 xv = *reinterpret_cast<const float2 *>(xr + ch);
                const uint32_t o = pack_bf16(xv.x + beta_l * lacc[nt][2 * h], xv.y + beta_l * lacc[nt][2 * h + 1]);
                *reinterpret_cast<uint32_t *>(sm + L.q + sw128_offset(trow, nt) + 4 * q4) = o;
            }
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        tma_store_4d(&mO, base + L.q, 0, c0, r0, sl);
        bulk_commit();
        bulk_wait_read0();
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ===========================================================================
// host side
// ===========================================================================
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D map over [S][n][64] bf16, box {64, 64 tokens, 1}.
bool make_map_tokens(CUtensorMap *m, const void *ptr, int S, int n) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)n, (cuuint64_t)S};
    cuuint64_t strides[2] = {(cuuint64_t)kRow, (cuuint64_t)n * kRow};
    cuuint32_t box[3] = {64, (cuuint32_t)kSub, 1}, es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over [S][H][W][64] bf16, box {64, bw, bh, 1}.
bool make_map_grid(CUtensorMap *m, const void *ptr, int S, int H, int W, int bh, int bw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)S};
    cuuint64_t strides[3] = {(cuuint64_t)kRow, (cuuint64_t)W * kRow, (cuuint64_t)H * W * kRow};
    cuuint32_t box[4] = {64, (cuuint32_t)bw, (cuuint32_t)bh, 1}, es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit once per device (and again
// only if a larger size is asked for), so calls made during stream capture
// do not touch function attributes.
template <typename Kern>
cudaError_t set_smem(Kern k, int slot, int bytes) {
    static std::mutex mu;
    static int done[4][64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[slot][dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[slot][dev] = bytes;
    return e;
}

uint32_t pow2_cols(int cols) {
    uint32_t c = 32;
    while ((int)c < cols) c <<= 1;
    return c;
}

}  // namespace

// Tile shape of the epilogue: th x tw = 128 tokens, both multiples of 4;
// fewest tiles, ties to the squarer shape.
void tc_tile_shape(int H, int W, int *th, int *tw) {
    static const int shapes[4][2] = {{8, 16}, {16, 8}, {4, 32}, {32, 4}};
    long best = -1;
    for (auto &s : shapes) {
        const long t = (long)((H + s[0] - 1) / s[0]) * ((W + s[1] - 1) / s[1]);
        if (best < 0 || t < best) {
            best = t;
            *th = s[0];
            *tw = s[1];
        }
    }
}

cudaError_t launch_tc(const Problem &p, cudaStream_t st, int stage) {
    TcParams t{};
    t.slices = p.slices; t.heads = p.heads; t.H = p.H; t.W = p.W; t.n = p.n; t.T = p.T;
    t.relu = p.relu; t.wmode = p.wmode; t.hidden = p.hidden; t.eps = p.eps; t.alpha = p.alpha;
    for (int k = 0; k < LISA_MAX_T; ++k) t.w[k] = p.w[k];
    t.W1 = p.W1; t.b1 = p.b1; t.W2 = p.W2; t.b2 = p.b2; t.K = p.K;
    t.chunks = p.chunks; t.chunk = p.chunk; t.cl = p.tc_cluster; t.parts = p.chunks / p.tc_cluster;
    tc_tile_shape(p.H, p.W, &t.th, &t.tw);
    t.tiles_r = (p.H + t.th - 1) / t.th;
    t.tiles_c = (p.W + t.tw - 1) / t.tw;
    const bool mlp = p.wmode == LISA_W_MLP;
    t.n_umat = mlp ? p.T - 1 : 1;
    t.epi_rows = 64 * t.n_umat + 16;
    t.n_mlp = mlp ? (p.hidden + 15) / 16 * 16 : 0;
    t.s_part = p.s_part; t.part = p.tc_part; t.bepi = p.tc_bepi; t.w1img = p.tc_w1img; t.err = p.err;

    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg{};
    cfg.stream = st;
    cfg.attrs = attrs;
    cudaError_t err = cudaSuccess;

    // 1. keysum
    if (stage < 0 || stage == 0) {
        cfg.gridDim = dim3((unsigned)(p.slices * p.chunks));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.numAttrs = 0;
        err = cudaLaunchKernelEx(&cfg, tc_keysum_kernel, t);
        if (err != cudaSuccess) return err;
    }
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    // 2. stats
    if (stage < 0 || stage == 1) {
        CUtensorMap mq, mk, mv;
        if (!make_map_tokens(&mq, p.Q, p.slices, p.n) || !make_map_tokens(&mk, p.K, p.slices, p.n) ||
            !make_map_tokens(&mv, p.V, p.slices, p.n))
            return cudaErrorInvalidValue;
        const int smem = kStages * kStageBytes + 1024;
        if ((err = set_smem(tc_stats_kernel, 0, smem)) != cudaSuccess) return err;
        cfg.gridDim = dim3((unsigned)(p.slices * p.chunks));
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        attrs[1].id = cudaLaunchAttributeClusterDimension;
        attrs[1].val.clusterDim.x = (unsigned)t.cl;
        attrs[1].val.clusterDim.y = 1;
        attrs[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        err = cudaLaunchKernelEx(&cfg, tc_stats_kernel, mq, mk, mv, t);
        if (err != cudaSuccess) return err;
    }
    // 3. recur
    if (stage < 0 || stage == 2) {
        cfg.gridDim = dim3((unsigned)(p.slices * kRecurRowBlocks));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, tc_recur_kernel, t);
        if (err != cudaSuccess) return err;
    }
    // 4. epilogue
    if (stage < 0 || stage == 3) {
        CUtensorMap mq, mkh, mvh, mkt, mo;
        if (!make_map_grid(&mq, p.Q, p.slices, p.H, p.W, t.th, t.tw) ||
            !make_map_grid(&mkh, p.K, p.slices, p.H, p.W, t.th + 2, t.tw + 2) ||
            !make_map_grid(&mvh, p.V, p.slices, p.H, p.W, t.th + 2, t.tw + 2) ||
            !make_map_grid(&mkt, p.K, p.slices, p.H, p.W, t.th, t.tw) ||
            !make_map_grid(&mo, p.O, p.slices, p.H, p.W, t.th, t.tw))
            return cudaErrorInvalidValue;
        const EpiLayout L = epi_layout(t.th, t.tw, t.epi_rows, t.n_mlp, mlp);
        const int smem = (int)L.total + 1024;
        if ((err = set_smem(tc_epilogue_kernel, 1, smem)) != cudaSuccess) return err;
        const uint32_t cols = pow2_cols(t.epi_rows + t.n_mlp);
        cfg.gridDim = dim3((unsigned)(p.slices * t.tiles_r * t.tiles_c));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = smem;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, tc_epilogue_kernel, mq, mkh, mvh, mkt, mo, t, cols);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

const char *const kTcStageNames[kTcStages] = {"tc_keysum", "tc_stats", "tc_recur", "tc_epilogue"};

}  // namespace lisa
