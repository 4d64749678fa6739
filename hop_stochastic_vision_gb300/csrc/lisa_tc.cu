// lisa_tc.cu -- tensor-core kernel chain of the LiSA forward layer for bf16
// layers with d_h = d_v = 64 on sm_103a.
//
// "note" below is the reading note of "LiSA: Linear Stochastic Attention for
// Long-Range Visual Modeling" (arXiv 2611.04216v2).  Per (batch, head)
// slice the layer needs the key sum s [note §2.2], the statistics
// U_1 = K^T V and M = K^T Q~ [note §2.3, paper Eq. 8], the recurrence
// U_k = M U_(k-1), and a per-token epilogue [note §2.4].  Two chains:
//
//  fused (a slice's chunks fit one thread-block cluster, <= 8 CTAs):
//   1. stats   each CTA streams its token chunk with TMA: its K rows stay
//              resident in shared memory; the cluster all-reduces s in
//              distributed shared memory; Q~_j = Q_j / (Q_j.s + eps) is formed
//              in shared memory and one tcgen05 MMA chain per CTA computes
//              [V | Q~]^T K = [U_1^T ; M^T] (128 x 64 fp32 in TMEM); the
//              cluster sums the chunk results (fixed order) and runs the
//              recurrence U_k^T = U_(k-1)^T M^T on its rows, writing the
//              epilogue's B operand [sum_k w_k U_k^T | s_hi | s_lo] in bf16.
//   2. epilogue (below).
//
//  split (longer slices, more chunks than a cluster holds):
//   1. keysum  s partials;  2. stats  cluster partials of [U_1^T ; M^T];
//   3. recur   reduction, recurrence and B operand;  4. epilogue.
//
//  epilogue: persistent CTAs walk 128-token tiles of the grid (2 x 8-token
//   blocks), double-buffering the TMA loads of the next tile.  tcgen05 forms
//   Q [U | s] (and [Q | K] W1^T for per-token weights) in TMEM; each warp runs
//   the 3x3 local branch of one 2 x 8 block on the legacy mma.sync path
//   (scores against the 4 x 10 key window, masked softmax, weights times V)
//   and reads the block's TMEM rows straight into the same fragment layout
//   (tcgen05.ld 16x256b), so the alpha mix happens in registers; TMA stores
//   the tile.
//
// Kernels are chained with programmatic dependent launch: each one's
// prologue and input prefetch overlap the previous kernel's tail.  Shared-
// memory operands use the 128-byte swizzle TMA writes (a 64-bf16 token row is
// 128 bytes; 8 rows form a 1024-byte atom).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "lisa_internal.h"
#include "lisa_sm100.cuh"
#include "lisa_solve.cuh"
#include "lisa_tc_common.cuh"

namespace lisa {
namespace {

using namespace sm100;

constexpr int kSub = 64;                       // tokens per stats pipeline stage
constexpr int kSubBytes = kSub * kRow;         // 8 KB
constexpr int kStages = 3;                     // stats pipeline depth
constexpr int kRecurRowBlocks = 4;             // split recur: CTAs per slice
constexpr int kRedStride = 68;                 // fp32 row stride of reduction buffers
constexpr int kFusedMaxSub = 7;                // fused stats: resident K chunk <= 448 tokens
constexpr int kFusedWork = 72 * 1024;          // fused stats: minimum work area

struct TcParams {
    int slices, heads, H, W, n, T, relu, wmode, hidden;
    int k_raw;                       // the K operand of the split statistics takes no feature map
    int untruncated;                 // U-bar = beta (1-beta) (I - beta M)^-1 U_1 instead of the series
    float eps, beta;
    const float *alpha;
    float w[LISA_MAX_T];
    const float *W1, *b1, *W2, *b2;
    const void *K;
    int chunks, chunk, cl, parts;    // split-K plan; cluster size; cluster partials per slice
    int BR, BC;                      // epilogue tile = BR x BC blocks of 2 x 8 tokens
    int tiles_r, tiles_c, tiles;     // tiles per slice (rows, cols), total tiles
    int epi_nbepi;                   // epilogue B-operand buffers (1 or 2)
    int slot_cols;                   // TMEM columns per epilogue slot
    int n_umat, epi_rows, n_mlp;     // B operand: U blocks, rows, MLP width (multiple of 16)
    float *s_part;                   // [S][C][64] (split chain)
    float *part;                     // [S][P][128][64] (split chain)
    uint8_t *bepi;                   // [S][epi_rows][128] bf16, 128-B swizzled rows
    uint8_t *w1img;                  // [2][n_mlp][128] bf16 (W1 q-part | k-part), swizzled
    int *err;
};

// U_next[i][a] = sum_b U[i][b] Mt[b][a] for `rows` rows (fp32, row stride 64,
// 16-byte aligned).  A work item is one row and four consecutive columns; U
// and Mt are read as float4, so each shared load feeds four FMAs; b in order.
__device__ __forceinline__ void rows_times_mt(const float *U, const float *Mt, float *Un, int rows,
                                              int tid, int nthreads) {
    for (int item = tid; item < rows * 16; item += nthreads) {
        const int i = item >> 4, c4 = item & 15;
        const float4 *u4 = reinterpret_cast<const float4 *>(U + i * 64);
        const float4 *m4 = reinterpret_cast<const float4 *>(Mt) + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int b4 = 0; b4 < 16; ++b4) {
            const float4 u = u4[b4];
            const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 m = m4[(4 * b4 + r) * 16];
                acc.x = fmaf(uu[r], m.x, acc.x);
                acc.y = fmaf(uu[r], m.y, acc.y);
                acc.z = fmaf(uu[r], m.z, acc.z);
                acc.w = fmaf(uu[r], m.w, acc.w);
            }
        }
        reinterpret_cast<float4 *>(Un + i * 64)[c4] = acc;
    }
}

// ------------------------------------------------------- shared stats steps
// Q~_j = Q_j / (Q_j . s + eps) in place for the 64 tokens of a stage (128
// threads, two per token, 32 features each); ReLU on load when asked.
__device__ __forceinline__ void form_qtilde(uint8_t *Qb, const float *s, float eps, int relu,
                                            int tid) {
    const int j = tid >> 1, h = tid & 1;
    uint4 q[4];
    float part[4] = {0.f, 0.f, 0.f, 0.f};   // one partial sum per 16-byte chunk
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int chunk = 4 * h + k;
        q[k] = *reinterpret_cast<uint4 *>(Qb + sw128_offset(j, chunk));
        if (relu) q[k] = relu4(q[k]);
        const uint32_t w4[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            part[k] = fmaf(bf16_lo(w4[e]), s[chunk * 8 + 2 * e], part[k]);
            part[k] = fmaf(bf16_hi(w4[e]), s[chunk * 8 + 2 * e + 1], part[k]);
        }
    }
    float dot = (part[0] + part[1]) + (part[2] + part[3]);
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    const float r = 1.f / (dot + eps);
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

// TMEM lanes lane0 .. lane0 + 31 (this warp's quadrant; 64 fp32 columns) ->
// shared rows `stride` floats apart: thread `lane` writes row 32 w + lane of
// `dst`.
__device__ __forceinline__ void tmem_rows_to_smem(uint32_t tmem, float *dst0, int w, int lane, int stride,
                                                  int lane0) {
    const int row = 32 * w + lane;
#pragma unroll
    for (int cb = 0; cb < 64; cb += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)lane0 << 16) + cb, r);
        tc_wait_ld();
        float4 *dst = reinterpret_cast<float4 *>(dst0 + row * stride + cb);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                 __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
    }
}

// W1 [hidden][128] -> two K-major bf16 images [n_mlp rows][64]: q-part, k-part.
__device__ __forceinline__ void put_w1_image(const TcParams &p, int tid, int nthreads) {
    for (int idx = tid; idx < 2 * p.n_mlp * 8; idx += nthreads) {
        const int half = idx / (p.n_mlp * 8), rem = idx % (p.n_mlp * 8);
        const int m = rem >> 3, chunk = rem & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[e] = m < p.hidden ? p.W1[(size_t)m * 2 * kD + half * kD + chunk * 8 + e] : 0.f;
        put_row_bf16(p.w1img + (size_t)half * p.n_mlp * kRow, m, v, chunk);
    }
}

// ===========================================================================
// fused stats: s, [U_1^T ; M^T] and the recurrence for one slice per cluster
// ===========================================================================
__device__ __forceinline__ void named_sync_compute() {
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the four compute warps only
}
// Barrier of the four compute warps that also ANDs a flag over them, so every
// thread takes the same branch after it.
__device__ __forceinline__ bool named_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Threads: warps 0-3 compute (prep, MMA issue, reductions), warp 4 produces
// the TMA loads and refills each ring stage as soon as its MMA completed.
constexpr int kStatsThreads = 160;

template <bool kUntruncated>
__global__ void __launch_bounds__(kStatsThreads) tc_stats_fused_kernel(const __grid_constant__ CUtensorMap mQ,
                                                                       const __grid_constant__ CUtensorMap mK,
                                                                       const __grid_constant__ CUtensorMap mV,
                                                                       TcParams p, int kres_bytes) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t kbar, full_bar[kStages], empty_bar[kStages], done_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ float s_loc[kD];
    __shared__ float s_sh[kD];
    __shared__ float s_red[16][kD + 1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sl = blockIdx.x / p.chunks, c = blockIdx.x % p.chunks;
    const uint32_t rank = cluster_rank();
    const int CL = p.cl;
    const int t0 = c * p.chunk;
    const int ntok = max(0, min(p.n, t0 + p.chunk) - t0);
    const int nsub = (ntok + kSub - 1) / kSub;
    const uint32_t base = smem_u32(sm);
    uint8_t *kres = sm;                                  // resident K rows of the chunk
    uint8_t *ring = sm + kres_bytes;                     // V | Q stages
    const uint32_t ring_addr = base + kres_bytes;
    constexpr int kStage = 2 * kSubBytes;

    if (tid == 0) {
        mbar_init(smem_u32(&kbar), 1);
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
    // Launched as a programmatic dependent of whatever kernel precedes it on the
    // stream: only set-up above this wait, which returns once that kernel has
    // finished and its writes (Q, K, V, or a previous call's use of the
    // workspace) are visible.  Dependents are released only after it.
    pdl_wait();
    if (blockIdx.x == 0 && tid == 0) *p.err = 0;
    pdl_launch_dependents();
    bool ok = true;

    if (warp == 4) {
        // ---------------- producer
        if (lane == 0) {
            mbar_arrive_expect_tx(smem_u32(&kbar), nsub * kSubBytes);
            for (int i = 0; i < nsub; ++i)
                tma_load_3d(base + i * kSubBytes, &mK, 0, t0 + i * kSub, sl, smem_u32(&kbar));
            // K gates the key sum and the cluster exchange: let it land first
            if (!mbar_wait(smem_u32(&kbar), 0)) record_error(p.err, kErrTimeoutLoad);
            for (int i = 0; i < kStages && i < nsub; ++i) {
                const uint32_t fb = smem_u32(&full_bar[i]);
                mbar_arrive_expect_tx(fb, kStage);
                tma_load_3d(ring_addr + i * kStage, &mV, 0, t0 + i * kSub, sl, fb);
                tma_load_3d(ring_addr + i * kStage + kSubBytes, &mQ, 0, t0 + i * kSub, sl, fb);
            }
        }
        __syncwarp();
        cluster_sync();                                  // (A) s exchange
        if (lane == 0) {
            for (int i = kStages; i < nsub; ++i) {
                const int st = i % kStages;
                // the MMA of sub-chunk i - kStages must have read the stage
                if (!mbar_wait(smem_u32(&empty_bar[st]), ((i - kStages) / kStages) & 1)) {
                    record_error(p.err, kErrTimeoutMma);
                    break;
                }
                const uint32_t fb = smem_u32(&full_bar[st]);
                mbar_arrive_expect_tx(fb, kStage);
                tma_load_3d(ring_addr + st * kStage, &mV, 0, t0 + i * kSub, sl, fb);
                tma_load_3d(ring_addr + st * kStage + kSubBytes, &mQ, 0, t0 + i * kSub, sl, fb);
            }
        }
        __syncwarp();
    } else {
        // ---------------- key sum (ReLU in place), then cluster all-reduce
        if (!mbar_wait(smem_u32(&kbar), 0)) {
            record_error(p.err, kErrTimeoutLoad);
            ok = false;
        }
        {
            const int cg = tid & 7, jl = tid >> 3;   // 16 token lanes x 8 feature chunks
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            for (int j0 = jl; j0 < nsub * kSub; j0 += 64) {   // four tokens per thread in flight
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const uint4 *>(kres + sw128_offset(j0 + 16 * u, cg));
                if (p.relu) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[u] = relu4(v[u]);
                        *reinterpret_cast<uint4 *>(kres + sw128_offset(j0 + 16 * u, cg)) = v[u];
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] += bf16_lo(w4[e]);
                        acc[2 * e + 1] += bf16_hi(w4[e]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s_red[jl][cg * 8 + e] = acc[e];
        }
        named_sync_compute();
        if (tid < kD) {
            float s = 0.f;
            for (int r = 0; r < 16; ++r) s += s_red[r][tid];
            s_loc[tid] = s;
        }
        fence_proxy_async();      // K's ReLU (generic proxy) before the MMAs read it
        cluster_sync();           // (A)
        if (tid < kD) {
            const uint32_t a = smem_u32(&s_loc[tid]);
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < CL) v[q] = ld_dsmem(map_rank(a, (uint32_t)q));
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < CL) s += v[q];
            s_sh[tid] = s;
        }
        named_sync_compute();

        // ---------------- [V | Q~]^T K over the chunk on tcgen05
        constexpr uint32_t idesc = make_idesc_bf16(128, 64, true, true);
        ok = named_sync_and(ok);
        for (int i = 0; i < nsub && ok; ++i) {
            const int st = i % kStages;
            if (!mbar_wait(smem_u32(&full_bar[st]), (i / kStages) & 1)) {
                record_error(p.err, kErrTimeoutLoad);
                ok = false;
            }
            if (!named_sync_and(ok)) break;
            form_qtilde(ring + st * kStage + kSubBytes, s_sh, p.eps, p.relu, tid);
            fence_proxy_async();
            named_sync_compute();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t vaddr = ring_addr + st * kStage;
                const uint32_t kaddr = base + i * kSubBytes;
#pragma unroll
                for (int ks = 0; ks < kSub / 16; ++ks) {
                    const uint64_t ad = make_desc_sw128(vaddr + ks * 2048, kSubBytes, 1024);
                    const uint64_t bd = make_desc_sw128(kaddr + ks * 2048, 1024, 1024);
                    tc_mma(tmem, ad, bd, idesc, (i | ks) != 0);
                }
                tc_commit(smem_u32(&empty_bar[st]));
            }
        }
        if (tid == 0) tc_commit(smem_u32(&done_bar));
        if (!mbar_wait(smem_u32(&done_bar), 0)) record_error(p.err, kErrTimeoutMma);
        tc_fence_after();
    }

    // ---- cluster reduction (fixed rank order): rank q sums rows q, q + CL, ...
    // and pushes each reduced M^T row into every CTA's copy of M^T; its own
    // U_1^T rows stay local.
    float *red = reinterpret_cast<float *>(sm);                    // [128][68]
    float *Mt = reinterpret_cast<float *>(sm + 36 * 1024);         // [64][kMS], filled by the owners
    float *Ucur = reinterpret_cast<float *>(sm + 54 * 1024);       // [my_u][kUS]
    const int my_u = (64 - (int)rank + CL - 1) / CL;               // own rows e < 64
    if (CL == 1) {
        // a slice in one CTA: no reduction, the rows go straight to U_1^T and M^T
        if (warp < 4) tmem_rows_to_smem(tmem, warp < 2 ? Ucur : Mt, warp & 1, lane, warp < 2 ? kUS : kMS, 32 * warp);
        tc_fence_before();
        __syncthreads();
    } else {
    if (warp < 4) tmem_rows_to_smem(tmem, red, warp, lane, kRedStride, 32 * warp);
    tc_fence_before();
    cluster_sync();                                                // (B)
    {
        const uint32_t red_addr = smem_u32(red);
        const uint32_t mt_addr = smem_u32(Mt);
        const int my_rows = (128 - (int)rank + CL - 1) / CL;
        for (int item = tid; item < my_rows * 16; item += kStatsThreads) {
            const int k = item >> 4, f = item & 15;
            const int rr = (int)rank + CL * k;
            const float4 v = cluster_sum4(red_addr + (uint32_t)(rr * kRedStride + 4 * f) * 4u, CL);
            if (rr < 64) {
                reinterpret_cast<float4 *>(Ucur + k * kUS)[f] = v;
            } else {
                const uint32_t dst = mt_addr + (uint32_t)((rr - 64) * kMS + 4 * f) * 4u;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < CL) st_dsmem4(map_rank(dst, (uint32_t)q), v);
            }
        }
    }
    cluster_sync();                                                // (C) M^T complete everywhere
    }
    if (kUntruncated) {
        // own rows of U_1^T become those of ((I - beta M)^-1 U_1)^T: A = I - beta M
        // in place of M^T (element (a, b) at Mt[b][a]), the own U_1 columns as R
        for (int idx = tid; idx < 64 * 64; idx += kStatsThreads) {
            const int b = idx >> 6, a = idx & 63;
            Mt[b * kMS + a] = (a == b ? 1.f : 0.f) - p.beta * Mt[b * kMS + a];
        }
        __syncthreads();
        constexpr int kW = kStatsThreads / 32;
        if (my_u <= 16)   // clusters of 4 or more CTAs: at most 80 columns
            solve_walk_system<kW, (80 + kW - 1) / kW>(Mt, kMS, Ucur, kUS, 64, my_u, &s_red[0][0], tid);
        else
            solve_walk_system<kW, (128 + kW - 1) / kW>(Mt, kMS, Ucur, kUS, 64, my_u, &s_red[0][0], tid);
    }

    // ---- U_k^T = U_(k-1)^T M^T on the own rows; B operand rows
    float *Unext = reinterpret_cast<float *>(sm);                  // [my_u][kUS]
    float *Fold = reinterpret_cast<float *>(sm + 18 * 1024);       // [my_u][kUS]
    const bool folded = (p.wmode != LISA_W_MLP);
    uint8_t *img = p.bepi + (size_t)sl * p.epi_rows * kRow;
    // k = 1: the fold starts at w_1 U_1 (or U_1's rows go out); then U_k = U_(k-1) M^T
    // on the tensor path into the other buffer, with the fold updated from the
    // result fragments
    if (folded) {
        const float w1 = p.T > 1 ? p.w[1] : 0.f;   // T = 1: no hop terms, the fold stays zero
        for (int item = tid; item < my_u * 16; item += kStatsThreads) {
            const float4 u = reinterpret_cast<const float4 *>(Ucur + (item >> 4) * kUS)[item & 15];
            reinterpret_cast<float4 *>(Fold + (item >> 4) * kUS)[item & 15] =
                make_float4(w1 * u.x, w1 * u.y, w1 * u.z, w1 * u.w);
        }
    } else {
        for (int item = tid; item < my_u * 8; item += kStatsThreads) {
            const int i = item >> 3, chunk = item & 7;
            put_row_bf16(img, (int)rank + CL * i, Ucur + i * kUS + chunk * 8, chunk);
        }
    }
    __syncthreads();
    float *Ua = Ucur, *Ub = Unext;
    for (int k = 2; k < p.T; ++k) {
        if (warp < 4) rows_times_mt_tf32(Ua, Mt, Ub, my_u, warp, lane, 4, folded ? Fold : nullptr, p.w[k]);
        __syncthreads();
        if (!folded)
            for (int item = tid; item < my_u * 8; item += kStatsThreads) {
                const int i = item >> 3, chunk = item & 7;
                put_row_bf16(img, (k - 1) * kD + (int)rank + CL * i, Ub + i * kUS + chunk * 8, chunk);
            }
        float *tmp = Ua;
        Ua = Ub;
        Ub = tmp;
    }
    if (folded)
        for (int item = tid; item < my_u * 8; item += kStatsThreads) {
            const int i = item >> 3, chunk = item & 7;
            put_row_bf16(img, (int)rank + CL * i, Fold + i * kUS + chunk * 8, chunk);
        }
    if (rank == 0) put_s_rows(img, p.n_umat * kD, s_sh, tid);
    if (!folded && sl == 0 && rank == 0) put_w1_image(p, tid, kStatsThreads);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ===========================================================================
// split chain: keysum, stats (cluster partials), recur
// ===========================================================================
__global__ void __launch_bounds__(256) tc_keysum_kernel(TcParams p) {
    __shared__ float red[32][kD + 1];
    const int sl = blockIdx.x / p.chunks, c = blockIdx.x % p.chunks;
    pdl_wait();   // first kernel of the chain: the preceding kernel's writes are visible after this
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.err = 0;
    pdl_launch_dependents();
    const int t0 = c * p.chunk, t1 = min(p.n, t0 + p.chunk);
    const int cg = threadIdx.x & 7, j0 = threadIdx.x >> 3;
    const uint4 *K = static_cast<const uint4 *>(p.K) + (size_t)sl * p.n * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    // every thread keeps the loads of a 512-token batch in flight together
    for (int jb = t0 + j0; jb < t1; jb += 512) {
        uint4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int j = jb + 32 * u;
            v[u] = j < t1 ? __ldg(K + (size_t)j * 8 + cg) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const uint4 x = p.relu ? relu4(v[u]) : v[u];
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += bf16_lo(w4[e]);
                acc[2 * e + 1] += bf16_hi(w4[e]);
            }
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

__device__ __forceinline__ void split_issue_loads(const CUtensorMap *mQ, const CUtensorMap *mK,
                                                  const CUtensorMap *mV, uint32_t stage_base,
                                                  uint32_t bar, int tok, int sl) {
    mbar_arrive_expect_tx(bar, 3 * kSubBytes);
    tma_load_3d(stage_base, mV, 0, tok, sl, bar);
    tma_load_3d(stage_base + kSubBytes, mQ, 0, tok, sl, bar);
    tma_load_3d(stage_base + 2 * kSubBytes, mK, 0, tok, sl, bar);
}

__global__ void __launch_bounds__(kStatsThreads) tc_stats_split_kernel(const __grid_constant__ CUtensorMap mQ,
                                                                       const __grid_constant__ CUtensorMap mK,
                                                                       const __grid_constant__ CUtensorMap mV,
                                                                       TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], done_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ float s_sh[kD];
    constexpr int kStage = 3 * kSubBytes;

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

    if (warp == 4) {
        // ---------------- producer: inputs do not depend on the earlier kernels
        if (lane == 0) {
            for (int i = 0; i < nsub; ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(smem_u32(&empty_bar[st]), ((i - kStages) / kStages) & 1)) {
                    record_error(p.err, kErrTimeoutMma);
                    break;
                }
                split_issue_loads(&mQ, &mK, &mV, base + st * kStage, smem_u32(&full_bar[st]), t0 + i * kSub, sl);
            }
        }
        __syncwarp();
    } else {
        pdl_wait();  // s partials are complete
        if (tid < kD) {
            s_sh[tid] = sum_partials(p.s_part + (size_t)sl * p.chunks * kD, p.chunks, kD, tid);
        }
        named_sync_compute();
        constexpr uint32_t idesc = make_idesc_bf16(128, 64, true, true);
        bool ok = true;
        for (int i = 0; i < nsub; ++i) {
            const int st = i % kStages;
            if (!mbar_wait(smem_u32(&full_bar[st]), (i / kStages) & 1)) {
                record_error(p.err, kErrTimeoutLoad);
                ok = false;
            }
            if (!named_sync_and(ok)) break;
            uint8_t *Vb = sm + st * kStage;
            if (p.relu && !p.k_raw) relu_smem(Vb + 2 * kSubBytes, kSubBytes, tid, 128);
            form_qtilde(Vb + kSubBytes, s_sh, p.eps, p.relu, tid);
            fence_proxy_async();
            named_sync_compute();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t vaddr = base + st * kStage;
                const uint32_t kaddr = vaddr + 2 * kSubBytes;
#pragma unroll
                for (int ks = 0; ks < kSub / 16; ++ks) {
                    const uint64_t ad = make_desc_sw128(vaddr + ks * 2048, kSubBytes, 1024);
                    const uint64_t bd = make_desc_sw128(kaddr + ks * 2048, 1024, 1024);
                    tc_mma(tmem, ad, bd, idesc, (i | ks) != 0);
                }
                tc_commit(smem_u32(&empty_bar[st]));
            }
        }
        if (tid == 0) tc_commit(smem_u32(&done_bar));
        if (!mbar_wait(smem_u32(&done_bar), 0)) record_error(p.err, kErrTimeoutMma);
        tc_fence_after();
    }

    float *red = reinterpret_cast<float *>(sm);
    if (warp < 4) tmem_rows_to_smem(tmem, red, warp, lane, kRedStride, 32 * warp);
    tc_fence_before();
    cluster_sync();
    const uint32_t rank = cluster_rank();
    const int CL = p.cl;
    float *out = p.part + ((size_t)sl * p.parts + c / CL) * 128 * kD;
    const int my_rows = (128 - (int)rank + CL - 1) / CL;
    const uint32_t red_addr = smem_u32(red);
    for (int item = tid; item < my_rows * 16; item += kStatsThreads) {
        const int rr = (int)rank + CL * (item >> 4);
        const int f = item & 15;
        const uint32_t off = (uint32_t)(rr * kRedStride + 4 * f) * 4u;
        reinterpret_cast<float4 *>(out + rr * kD)[f] = cluster_sum4(red_addr + off, CL);
    }
    cluster_sync();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

__global__ void __launch_bounds__(256) tc_recur_kernel(TcParams p) {
    __shared__ __align__(16) float Mt[kD][kD];     // M^T [b][a]
    __shared__ __align__(16) float Ut[16][kD];     // this CTA's 16 rows of U_k^T
    __shared__ __align__(16) float Un[16][kD];
    __shared__ __align__(16) float Fold[16][kD];
    __shared__ float s_sh[kD];
    __shared__ float fac[3 * kD];                  // solve scratch (untruncated walk)
    const int tid = threadIdx.x;
    const int sl = blockIdx.x / kRecurRowBlocks, rb = blockIdx.x % kRecurRowBlocks;
    pdl_launch_dependents();
    pdl_wait();
    const float4 *part = reinterpret_cast<const float4 *>(p.part + (size_t)sl * p.parts * 128 * kD);
    // M^T: 1024 float4, 4 per thread; each partial's loads issued before the sums
    {
        float4 acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int q = 0; q < p.parts; ++q) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = part[((size_t)q * 128 + kD) * 16 + tid + 256 * u];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc[u].x += v[u].x; acc[u].y += v[u].y; acc[u].z += v[u].z; acc[u].w += v[u].w;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) reinterpret_cast<float4 *>(&Mt[0][0])[tid + 256 * u] = acc[u];
    }
    {   // own 16 rows of U_1^T: 256 float4, one per thread
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int q = 0; q < p.parts; ++q) {
            const float4 v = part[((size_t)q * 128 + 16 * rb) * 16 + tid];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4 *>(&Ut[0][0])[tid] = acc;
        reinterpret_cast<float4 *>(&Fold[0][0])[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < kD) {
        s_sh[tid] = sum_partials(p.s_part + (size_t)sl * p.chunks * kD, p.chunks, kD, tid);
    }
    __syncthreads();
    if (p.untruncated) {   // own rows of U_1^T -> those of ((I - beta M)^-1 U_1)^T
        for (int idx = tid; idx < kD * kD; idx += 256) {
            const int b = idx >> 6, a = idx & 63;
            Mt[b][a] = (a == b ? 1.f : 0.f) - p.beta * Mt[b][a];
        }
        __syncthreads();
        solve_walk_system<8, 10>(&Mt[0][0], kD, &Ut[0][0], kD, kD, 16, fac, tid);
    }
    const bool folded = (p.wmode != LISA_W_MLP);
    uint8_t *img = p.bepi + (size_t)sl * p.epi_rows * kRow;
    for (int k = 1; k < p.T; ++k) {
        if (k > 1) {
            rows_times_mt(&Ut[0][0], &Mt[0][0], &Un[0][0], 16, tid, 256);
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
    if (rb == 0) put_s_rows(img, p.n_umat * kD, s_sh, tid);
    if (!folded && sl == 0 && rb == 0) put_w1_image(p, tid, 256);
}

// ===========================================================================
// epilogue
// ===========================================================================
// Threads: eight compute warps, each owning one 2 x 8 token block of the
// 128-token tile, and one control warp whose lane 0 issues every TMA load and
// tensor-core MMA.  Tiles move through kSlots input slots; mbarriers carry
// every hand-off, so no block-wide barrier sits inside the tile loop:
//   qk_full, v_full    a slot's Q + K halo (+ the tile's K rows) / V halo landed
//   qrelu              the compute warps wrote the ReLU'd Q (and K rows) back
//   mma_full           the tile's products are in its TMEM slot
//   qk_empty, v_empty  the compute warps no longer read the slot's Q/K, V
//   tmem_empty         the compute warps have read their rows of the TMEM slot
//   b_full, b_free     a B-operand buffer landed / its last MMA completed
// Each compute warp stages its 2 x 8 output block in its own two buffers and
// stores it with TMA itself.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * (kEpiWarps + 1);
constexpr int kMlpKSteps = LISA_MAX_HIDDEN / 16;   // m16n8k16 steps over the MLP's hidden units
// Per-lane constants of the MLP head, [2 kMlpKSteps][32 lanes] of 16 bytes:
// entry kk < kMlpKSteps holds the W2^T B fragments of k-step kk (hi, hi, lo, lo),
// entry kMlpKSteps + kk the b1 values of the lane's columns in f8 = 2 kk, 2 kk + 1.
constexpr uint32_t kMlpConstBytes = 2u * kMlpKSteps * 32u * 16u;
constexpr uint32_t kOutBuf = 16 * kRow;   // one warp's 2 x 8 output block

struct EpiLayout {
    uint32_t q[2], kh[2], vh[2], kt[2], bepi[2], w1, mlpc, out, total;
};

__host__ __device__ inline uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

__host__ __device__ inline EpiLayout epi_layout(int BR, int BC, int epi_rows, int n_mlp, bool mlp, int slots,
                                                int nbepi) {
    EpiLayout L{};
    const uint32_t halo = align1k((uint32_t)(2 * BR + 2) * (8 * BC + 2) * kRow);
    uint32_t off = 0;
    for (int s = 0; s < 2; ++s) {
        if (s < slots) {
            L.q[s] = off; off += 128 * kRow;
            L.kh[s] = off; off += halo;
            L.vh[s] = off; off += halo;
            L.kt[s] = off; if (mlp) off += 128 * kRow;
        } else {
            L.q[s] = L.q[0]; L.kh[s] = L.kh[0]; L.vh[s] = L.vh[0]; L.kt[s] = L.kt[0];
        }
    }
    for (int b = 0; b < 2; ++b) {
        if (b < nbepi) {
            L.bepi[b] = off;
            off += align1k((uint32_t)epi_rows * kRow);
        } else {
            L.bepi[b] = L.bepi[0];
        }
    }
    L.w1 = off; if (mlp) off += align1k(2u * n_mlp * kRow);
    L.mlpc = off; if (mlp) off += kMlpConstBytes;
    L.out = off; off += kEpiWarps * 2 * kOutBuf;
    L.total = off;
    return L;
}

struct TileCoord {
    int sl, r0, c0;
};
__device__ __forceinline__ TileCoord tile_coord(const TcParams &p, int t) {
    const int per = p.tiles_r * p.tiles_c;
    TileCoord tc;
    tc.sl = t / per;
    const int rem = t % per;
    tc.r0 = (rem / p.tiles_c) * (2 * p.BR);
    tc.c0 = (rem % p.tiles_c) * (8 * p.BC);
    return tc;
}

struct EpiBars {
    uint64_t qk_full[2], v_full[2], qrelu[2], mma_full[2], qk_empty[2], v_empty[2], tmem_empty[2];
    uint64_t b_full[2], b_free[2], w1;
};

template <bool kMlp, int kSlots, int kMinBlocks>
__global__ void __launch_bounds__(kEpiThreads, kMinBlocks)
    tc_epilogue_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKh,
                       const __grid_constant__ CUtensorMap mVh, const __grid_constant__ CUtensorMap mKt,
                       const __grid_constant__ CUtensorMap mO, TcParams p, uint32_t tmem_cols) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) EpiBars bar;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool mlp = kMlp;
    const int BR = p.BR, BC = p.BC, hw = 8 * BC + 2;
    const EpiLayout L = epi_layout(BR, BC, p.epi_rows, p.n_mlp, mlp, kSlots, p.epi_nbepi);
    const uint32_t base = smem_u32(sm);

    // contiguous run of tiles (consecutive tiles mostly share a slice); runs
    // differ in length by at most one tile
    const int t_begin = (int)((long long)blockIdx.x * p.tiles / gridDim.x);
    const int t_end = (int)((long long)(blockIdx.x + 1) * p.tiles / gridDim.x);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bar.qk_full[s]), 1);
            mbar_init(smem_u32(&bar.v_full[s]), 1);
            mbar_init(smem_u32(&bar.mma_full[s]), 1);
            mbar_init(smem_u32(&bar.qrelu[s]), kEpiWarps);
            mbar_init(smem_u32(&bar.qk_empty[s]), kEpiWarps);
            mbar_init(smem_u32(&bar.v_empty[s]), kEpiWarps);
            mbar_init(smem_u32(&bar.tmem_empty[s]), kEpiWarps);
            mbar_init(smem_u32(&bar.b_full[s]), 1);
            mbar_init(smem_u32(&bar.b_free[s]), 1);
        }
        mbar_init(smem_u32(&bar.w1), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    if (warp == kEpiWarps) {
        // ===================== control: TMA loads and tensor-core products
        if (lane == 0 && t_begin < t_end) {
            const uint32_t halo_tx = (uint32_t)(2 * BR + 2) * hw * kRow;
            auto load_qk = [&](int t, int s) {
                const TileCoord tc = tile_coord(p, t);
                const uint32_t b = smem_u32(&bar.qk_full[s]);
                mbar_arrive_expect_tx(b, (mlp ? 256u : 128u) * kRow + halo_tx);
                for (int bj = 0; bj < BC; ++bj) {
                    tma_load_4d(base + L.q[s] + bj * 16 * BR * kRow, &mQ, 0, tc.c0 + 8 * bj, tc.r0, tc.sl, b);
                    if (mlp)
                        tma_load_4d(base + L.kt[s] + bj * 16 * BR * kRow, &mKt, 0, tc.c0 + 8 * bj, tc.r0, tc.sl, b);
                }
                tma_load_4d(base + L.kh[s], &mKh, 0, tc.c0 - 1, tc.r0 - 1, tc.sl, b);
            };
            auto load_v = [&](int t, int s) {
                const TileCoord tc = tile_coord(p, t);
                const uint32_t b = smem_u32(&bar.v_full[s]);
                mbar_arrive_expect_tx(b, halo_tx);
                tma_load_4d(base + L.vh[s], &mVh, 0, tc.c0 - 1, tc.r0 - 1, tc.sl, b);
            };
            // the tiles' Q, K, V do not depend on the previous kernel
            for (int u = 0; u < kSlots && t_begin + u < t_end; ++u) {
                load_qk(t_begin + u, u);
                load_v(t_begin + u, u);
            }
            pdl_wait();   // the B operands (and the W1 image) come from the previous kernel
            if (mlp) {
                mbar_arrive_expect_tx(smem_u32(&bar.w1), 2u * p.n_mlp * kRow);
                bulk_load(base + L.w1, p.w1img, 2u * p.n_mlp * kRow, smem_u32(&bar.w1));
                if (!mbar_wait(smem_u32(&bar.w1), 0)) record_error(p.err, kErrTimeoutLoad);
            }
            const int nb = p.epi_nbepi;
            const uint32_t brow_bytes = (uint32_t)p.epi_rows * kRow;
            int cur_sl = -1, cur_b = 0, n_loads = 0;
            int commits[2] = {0, 0}, waited[2] = {0, 0};
            for (int t = t_begin, it = 0; t < t_end; ++t, ++it) {
                const int s = it % kSlots;
                const uint32_t ph = (uint32_t)(it / kSlots) & 1u;
                const int sl = tile_coord(p, t).sl;
                if (sl != cur_sl) {
                    // B operand of a new slice; its buffer's previous slice must be done
                    cur_b = n_loads % nb;
                    const int use = n_loads / nb;
                    if (use > 0) {
                        if (!mbar_wait(smem_u32(&bar.b_free[cur_b]), (uint32_t)(use - 1) & 1u))
                            record_error(p.err, kErrTimeoutMma);
                        waited[cur_b] = use;
                    }
                    const uint32_t b = smem_u32(&bar.b_full[cur_b]);
                    mbar_arrive_expect_tx(b, brow_bytes);
                    bulk_load(base + L.bepi[cur_b], p.bepi + (size_t)sl * brow_bytes, brow_bytes, b);
                    if (!mbar_wait(b, (uint32_t)use & 1u)) record_error(p.err, kErrTimeoutLoad);
                    ++n_loads;
                    cur_sl = sl;
                }
                if (!mbar_wait(smem_u32(&bar.qrelu[s]), ph)) record_error(p.err, kErrTimeoutLoad);
                if (it >= kSlots && !mbar_wait(smem_u32(&bar.tmem_empty[s]), ph ^ 1u))
                    record_error(p.err, kErrTimeoutMma);
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(s * p.slot_cols);
                const uint32_t qa = base + L.q[s], ba = base + L.bepi[cur_b];
                for (int r = 0; r < p.epi_rows; r += 256) {
                    const int N = min(256, p.epi_rows - r);
                    const uint32_t idesc = make_idesc_bf16(128, N, false, false);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc_mma(d + r, make_desc_sw128(qa + ks * 32, 16, 1024),
                               make_desc_sw128(ba + r * kRow + ks * 32, 16, 1024), idesc, ks > 0);
                }
                if (mlp) {
                    // hidden pre-activations [Q | K] W1^T next to the global products
                    const uint32_t idesc = make_idesc_bf16(128, p.n_mlp, false, false);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t a = base + (ks < 4 ? L.q[s] : L.kt[s]) + (ks & 3) * 32;
                        const uint32_t b = base + L.w1 + (ks < 4 ? 0u : (uint32_t)p.n_mlp * kRow) + (ks & 3) * 32;
                        tc_mma(d + p.epi_rows, make_desc_sw128(a, 16, 1024), make_desc_sw128(b, 16, 1024), idesc,
                               ks > 0);
                    }
                }
                tc_commit(smem_u32(&bar.mma_full[s]));
                if (t + 1 < t_end && tile_coord(p, t + 1).sl != sl) {
                    tc_commit(smem_u32(&bar.b_free[cur_b]));
                    ++commits[cur_b];
                }
                // refill this slot with tile it + kSlots as soon as the warps and the MMA let go of it
                if (t + kSlots < t_end) {
                    if (!mbar_wait(smem_u32(&bar.qk_empty[s]), ph)) record_error(p.err, kErrTimeoutLoad);
                    if (!mbar_wait(smem_u32(&bar.mma_full[s]), ph)) record_error(p.err, kErrTimeoutMma);
                    load_qk(t + kSlots, s);
                    if (!mbar_wait(smem_u32(&bar.v_empty[s]), ph)) record_error(p.err, kErrTimeoutLoad);
                    load_v(t + kSlots, s);
                }
            }
            // no commit may still be in flight when the CTA exits
            for (int b = 0; b < 2; ++b)
                if (commits[b] > waited[b] && !mbar_wait(smem_u32(&bar.b_free[b]), (uint32_t)waited[b] & 1u))
                    record_error(p.err, kErrTimeoutMma);
        }
        __syncwarp();
    } else {
        // ===================== compute: local branch, mix, store
        const int g = lane >> 2, q4 = lane & 3;
        // this warp's 2 x 8 block: TMEM lanes 16 blk .. 16 blk + 15 (inside its quadrant)
        const int blk = 2 * (warp & 3) + (warp >> 2);
        const int bi = blk % BR, bj = blk / BR;
        const uint32_t lane_base = (uint32_t)(16 * blk) << 16;

        // Per-lane constants of the local branch.  Window key kappa indexes the
        // 4 x 10 key window of the block: ka = kappa / 10, kb = kappa % 10.
        // Score element (j, e) of this lane: row g + 8 (e >> 1), key 8 j + 2 q + (e & 1).
        uint32_t win_mask = 0;   // bit j*4+e: key in the query's 3x3 window
        uint32_t ctr_mask = 0;   // bit j*4+e: key is the query token itself
#pragma unroll
        for (int j = 0; j < 5; ++j)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int kappa = 8 * j + 2 * q4 + b;
                const int ka = kappa / 10, kb = kappa % 10;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int du = ka - h, dv = kb - g;
                    if (du >= 0 && du <= 2 && dv >= 0 && dv <= 2) win_mask |= 1u << (j * 4 + 2 * h + b);
                    if (du == 1 && dv == 1) ctr_mask |= 1u << (j * 4 + 2 * h + b);
                }
            }
        float wbias[5][4];           // 0 inside the window, -inf outside (blocks off the grid border)
#pragma unroll
        for (int j = 0; j < 5; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) wbias[j][e] = ((win_mask >> (j * 4 + e)) & 1u) ? 0.f : -INFINITY;
        uint32_t koff[3], voff[3];   // halo rows of the ldmatrix loads (static per warp)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const int kk = 8 * (2 * pr + (lane >> 4)) + (lane & 7);       // scores: n-tile pairs
            const int kv = 16 * pr + (lane & 7) + 8 * ((lane >> 3) & 1);   // values: k-steps
            const int kk2 = kk < 40 ? kk : 0, kv2 = kv < 40 ? kv : 0;
            koff[pr] = (uint32_t)((2 * bi + kk2 / 10) * hw + 8 * bj + kk2 % 10);
            voff[pr] = (uint32_t)((2 * bi + kv2 / 10) * hw + 8 * bj + kv2 % 10);
        }
        const uint32_t qrow = (uint32_t)(16 * blk + (lane & 7) + 8 * ((lane >> 3) & 1));   // A-fragment row

        // Adaptive weights: the logits z = W2 h + b2 of the 16 rows are one
        // m16n8k16 product per 16 hidden units, h in the C-fragment layout the
        // TMEM read gives (which is also the A-fragment layout).  W2^T as B
        // fragments (k = hidden unit, n = walk length t) and b1 at this lane's
        // hidden columns depend on the lane only: compute warp 0 writes them to
        // a table once, every compute warp reads its lane's entries per tile.
        // W2 and h are each split into two bf16 terms (hi + lo), so the
        // product keeps ~16 significant bits.
        const uint32_t mlpc = base + L.mlpc + (uint32_t)lane * 16u;
        float b2r[2];
        if (mlp) {
            if (warp == 0) {
#pragma unroll
                for (int kk = 0; kk < kMlpKSteps; ++kk) {
                    uint32_t hi[2], lo[2];
                    float b1v[4];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int m0 = 16 * kk + 8 * hf + 2 * q4;
                        float x[2];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            x[c] = (g < p.T && m0 + c < p.hidden) ? p.W2[g * p.hidden + m0 + c] : 0.f;
                            b1v[2 * hf + c] = m0 + c < p.hidden ? p.b1[m0 + c] : 0.f;
                        }
                        hi[hf] = pack_bf16(x[0], x[1]);
                        lo[hf] = pack_bf16(x[0] - bf16_lo(hi[hf]), x[1] - bf16_hi(hi[hf]));
                    }
                    st_shared_v4(mlpc + (uint32_t)kk * 512u, hi[0], hi[1], lo[0], lo[1]);
                    st_shared_v4(mlpc + (uint32_t)(kMlpKSteps + kk) * 512u, __float_as_uint(b1v[0]),
                                 __float_as_uint(b1v[1]), __float_as_uint(b1v[2]), __float_as_uint(b1v[3]));
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) b2r[c] = 2 * q4 + c < p.T ? p.b2[2 * q4 + c] : 0.f;
            asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");   // the compute warps only
        }
        const uint32_t out_w = base + L.out + (uint32_t)warp * 2u * kOutBuf;
        const float c2 = 1.4426950408889634f * 0.125f;   // log2(e) / sqrt(64)

        TileCoord tc = tile_coord(p, t_begin);
        int alpha_sl = -1;   // the head's alpha is read from global memory once per slice
        float alpha = 0.f;
        for (int t = t_begin, it = 0; t < t_end; ++t, ++it) {
            if (it > 0) {   // next tile in row-major order of the slice's tile grid
                tc.c0 += 8 * BC;
                if (tc.c0 >= 8 * BC * p.tiles_c) {
                    tc.c0 = 0;
                    tc.r0 += 2 * BR;
                    if (tc.r0 >= 2 * BR * p.tiles_r) {
                        tc.r0 = 0;
                        ++tc.sl;
                    }
                }
            }
            const int s = it % kSlots;
            const uint32_t ph = (uint32_t)(it / kSlots) & 1u;
            if (tc.sl != alpha_sl) {
                alpha = p.alpha[tc.sl % p.heads];
                alpha_sl = tc.sl;
            }
            const uint32_t tl = tmem + (uint32_t)(s * p.slot_cols) + lane_base;

            // ---- the block's queries: A fragments, ReLU'd in registers and written
            // back (with the tile's K rows) for the tensor-core products
            if (!mbar_wait(smem_u32(&bar.qk_full[s]), ph)) record_error(p.err, kErrTimeoutLoad);
            const uint32_t qb = base + L.q[s];
            uint32_t a[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(qb + sw128_offset(qrow, 2 * ks + (lane >> 4)), a[ks][0], a[ks][1], a[ks][2], a[ks][3]);
            if (p.relu) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) a[ks][e] = relu2(a[ks][e]);
                    stsm_x4(qb + sw128_offset(qrow, 2 * ks + (lane >> 4)), a[ks][0], a[ks][1], a[ks][2], a[ks][3]);
                }
                if (mlp) {
                    const uint32_t kb = base + L.kt[s];
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t ad = kb + sw128_offset(qrow, 2 * ks + (lane >> 4));
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(ad, r0, r1, r2, r3);
                        stsm_x4(ad, relu2(r0), relu2(r1), relu2(r2), relu2(r3));
                    }
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.qrelu[s]));

            // ---- local branch scores: Q block (16 x 64) against its 4 x 10 key window
            float sc[5][4];
            {
                const uint32_t khb = base + L.kh[s];
#pragma unroll
                for (int j = 0; j < 5; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                    for (int pr = 0; pr < 3; ++pr) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(khb + sw128_offset(koff[pr], 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
                        if (p.relu) {
                            b0 = relu2(b0); b1 = relu2(b1); b2 = relu2(b2); b3 = relu2(b3);
                        }
                        mma_bf16_16816(sc[2 * pr], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
                        if (pr < 2) mma_bf16_16816(sc[2 * pr + 1], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.qk_empty[s]));

            float w0[2], wq[2][2];
            if (mlp) {
                // adaptive step weights of rows g, g+8 from the MLP hidden layer in TMEM
                if (!mbar_wait(smem_u32(&bar.mma_full[s]), ph)) record_error(p.err, kErrTimeoutMma);
                tc_fence_after();
                // z (C fragment): (row g, t = 2 q4, 2 q4 + 1), (row g + 8, same)
                float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < kMlpKSteps; ++kk) {
                    if (16 * kk >= p.n_mlp) break;
                    uint32_t hr[2][4];   // pre-activations of hidden columns 16 kk .. 16 kk + 15
                    tmem_ld_frag_nowait(tl + p.epi_rows + 16 * kk, hr[0]);
                    tmem_ld_frag_nowait(tl + p.epi_rows + 16 * kk + 8, hr[1]);
                    uint32_t wf[4], bw[4], ahi[4], alo[4];
                    ld_shared_v4(mlpc + (uint32_t)kk * 512u, wf[0], wf[1], wf[2], wf[3]);
                    ld_shared_v4(mlpc + (uint32_t)(kMlpKSteps + kk) * 512u, bw[0], bw[1], bw[2], bw[3]);
                    tc_wait_ld();
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        // A register r: hidden columns of f8 = 2 kk + (r >> 1), row g (r even) or g + 8
                        const int hf = r >> 1, e = 2 * (r & 1);
                        const float h0 = gelu_as7126(__uint_as_float(hr[hf][e]) + __uint_as_float(bw[2 * hf]));
                        const float h1 = gelu_as7126(__uint_as_float(hr[hf][e + 1]) + __uint_as_float(bw[2 * hf + 1]));
                        ahi[r] = pack_bf16(h0, h1);
                        alo[r] = pack_bf16(h0 - bf16_lo(ahi[r]), h1 - bf16_hi(ahi[r]));
                    }
                    mma_bf16_16816(z, ahi[0], ahi[1], ahi[2], ahi[3], wf[0], wf[1]);
                    mma_bf16_16816(z, alo[0], alo[1], alo[2], alo[3], wf[0], wf[1]);
                    mma_bf16_16816(z, ahi[0], ahi[1], ahi[2], ahi[3], wf[2], wf[3]);
                }
                // softmax over t < T across the four lanes of the row's quad
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float zz[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c) zz[c] = 2 * q4 + c < p.T ? z[2 * h + c] + b2r[c] : -INFINITY;
                    float zmax = fmaxf(zz[0], zz[1]);
                    zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, 1));
                    zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, 2));
#pragma unroll
                    for (int c = 0; c < 2; ++c) wq[h][c] = 2 * q4 + c < p.T ? expf(zz[c] - zmax) : 0.f;
                    float zs = wq[h][0] + wq[h][1];
                    zs += __shfl_xor_sync(0xffffffffu, zs, 1);
                    zs += __shfl_xor_sync(0xffffffffu, zs, 2);
                    const float zi = 1.f / zs;
                    wq[h][0] *= zi;
                    wq[h][1] *= zi;
                }
                // weight t of row h sits in lane (quad | t >> 1), element t & 1
                w0[0] = __shfl_sync(0xffffffffu, wq[0][0], lane & ~3);
                w0[1] = __shfl_sync(0xffffffffu, wq[1][0], lane & ~3);
            } else {
                w0[0] = w0[1] = p.w[0];
            }

            // ---- masked softmax over the window; the weight matrix also carries
            // alpha w_0 on the token itself, so P' V = (1 - alpha) l_i + alpha w_0 V_i
            float lacc[8][4];
            {
                const int gr0 = tc.r0 + 2 * bi - 1, gc0 = tc.c0 + 8 * bj - 1;   // grid position of window (0, 0)
                if (gr0 < 0 || gr0 + 3 >= p.H || gc0 < 0 || gc0 + 9 >= p.W) {
                    // block on the grid border: drop the window keys outside the grid
                    uint32_t mask = win_mask;
#pragma unroll
                    for (int j = 0; j < 5; ++j)
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const int kappa = 8 * j + 2 * q4 + b;
                            const int gr = gr0 + kappa / 10, gc = gc0 + kappa % 10;
                            if (gr < 0 || gr >= p.H || gc < 0 || gc >= p.W) mask &= ~(0x5u << (j * 4 + b));
                        }
#pragma unroll
                    for (int j = 0; j < 5; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[j][e] = ((mask >> (j * 4 + e)) & 1u) ? sc[j][e] * c2 : -INFINITY;
                } else {
#pragma unroll
                    for (int j = 0; j < 5; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[j][e] = fmaf(sc[j][e], c2, wbias[j][e]);
                }
                // row maxima and sums as balanced trees over the 10 elements of each row
                float mx[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float a0 = fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), a1 = fmaxf(sc[1][2 * h], sc[1][2 * h + 1]);
                    const float a2 = fmaxf(sc[2][2 * h], sc[2][2 * h + 1]), a3 = fmaxf(sc[3][2 * h], sc[3][2 * h + 1]);
                    const float a4 = fmaxf(sc[4][2 * h], sc[4][2 * h + 1]);
                    mx[h] = fmaxf(fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)), a4);
                }
                float sum[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                    if (mx[h] == -INFINITY) mx[h] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 5; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[j][e] = ex2_approx(sc[j][e] - mx[e >> 1]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float a0 = sc[0][2 * h] + sc[0][2 * h + 1], a1 = sc[1][2 * h] + sc[1][2 * h + 1];
                    const float a2 = sc[2][2 * h] + sc[2][2 * h + 1], a3 = sc[3][2 * h] + sc[3][2 * h + 1];
                    const float a4 = sc[4][2 * h] + sc[4][2 * h + 1];
                    sum[h] = ((a0 + a1) + (a2 + a3)) + a4;
                }
                float scale[2], self[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
                    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
                    scale[h] = sum[h] > 0.f ? __fdividef(1.f - alpha, sum[h]) : 0.f;
                    self[h] = alpha * w0[h];
                }
#pragma unroll
                for (int j = 0; j < 5; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[j][e] = fmaf(sc[j][e], scale[e >> 1], ((ctr_mask >> (j * 4 + e)) & 1u) ? self[e >> 1] : 0.f);

                if (!mbar_wait(smem_u32(&bar.v_full[s]), ph)) record_error(p.err, kErrTimeoutLoad);
                const uint32_t vhb = base + L.vh[s];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) lacc[nt][0] = lacc[nt][1] = lacc[nt][2] = lacc[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 3; ++ks) {
                    const int j0 = 2 * ks, j1 = 2 * ks + 1;
                    const uint32_t pa0 = pack_bf16(sc[j0][0], sc[j0][1]);
                    const uint32_t pa1 = pack_bf16(sc[j0][2], sc[j0][3]);
                    const uint32_t pa2 = j1 < 5 ? pack_bf16(sc[j1][0], sc[j1][1]) : 0u;
                    const uint32_t pa3 = j1 < 5 ? pack_bf16(sc[j1][2], sc[j1][3]) : 0u;
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vhb + sw128_offset(voff[ks], 2 * np + (lane >> 4)), b0, b1, b2, b3);
                        mma_bf16_16816(lacc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
                        mma_bf16_16816(lacc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.v_empty[s]));

            // ---- global branch from TMEM (fragment layout), mix, output block
            if (!mlp && !mbar_wait(smem_u32(&bar.mma_full[s]), ph)) record_error(p.err, kErrTimeoutMma);
            tc_fence_after();
            float acc[32], arq[2];
            {
                uint32_t rs[4], ru[32];
                tmem_ld_frag_nowait(tl + p.n_umat * kD, rs);   // Q.s_hi, Q.s_lo: columns held by lane q4 = 0
                tmem_ld_frag8_nowait(tl, ru);
                tc_wait_ld();
                const int src = lane & ~3;
                const float d0 = __shfl_sync(0xffffffffu, __uint_as_float(rs[0]) + __uint_as_float(rs[1]), src);
                const float d1 = __shfl_sync(0xffffffffu, __uint_as_float(rs[2]) + __uint_as_float(rs[3]), src);
                // alpha / (Q_i . s + eps): the global term is alpha Q~_i U = alpha (Q_i U) / (Q_i . s + eps)
                arq[0] = __fdividef(alpha, d0 + p.eps);
                arq[1] = __fdividef(alpha, d1 + p.eps);
                if (mlp) {
                    // walk length t = u + 1 weighs the product with U_(u+1)
                    float wu[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) wu[h] = __shfl_sync(0xffffffffu, wq[h][1], lane & ~3);
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[k] = wu[(k >> 1) & 1] * __uint_as_float(ru[k]);
#pragma unroll
                    for (int u = 1; u < LISA_MAX_T_MLP - 1; ++u) {
                        if (u >= p.n_umat) break;
                        tmem_ld_frag8_nowait(tl + u * kD, ru);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            wu[h] = __shfl_sync(0xffffffffu, wq[h][(u + 1) & 1], (lane & ~3) | ((u + 1) >> 1));
                        tc_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) acc[k] = fmaf(wu[(k >> 1) & 1], __uint_as_float(ru[k]), acc[k]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[k] = __uint_as_float(ru[k]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.tmem_empty[s]));

            const uint32_t ob = out_w + (uint32_t)(it & 1) * kOutBuf;
            if (lane == 0) bulk_wait_read<1>();   // the store that last read this buffer is done with it
            __syncwarp();
            // stmatrix: matrix m of a store is (nt0 + m / 2, rows 8 (m % 2) ..); lane l
            // addresses row l % 8 of matrix l / 8 (swizzled 16-byte chunk nt ^ row)
#pragma unroll
            for (int nt0 = 0; nt0 < 8; nt0 += 2) {
                uint32_t r[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int nt = nt0 + (m >> 1), h = m & 1;
                    r[m] = pack_bf16(fmaf(arq[h], acc[4 * nt + 2 * h], lacc[nt][2 * h]),
                                     fmaf(arq[h], acc[4 * nt + 2 * h + 1], lacc[nt][2 * h + 1]));
                }
                const uint32_t mrow = (uint32_t)(lane & 7), mm = (uint32_t)(lane >> 3);
                stsm_x4(ob + (8u * (mm & 1u) + mrow) * kRow + ((((uint32_t)nt0 + (mm >> 1)) ^ mrow) << 4), r[0], r[1],
                        r[2], r[3]);
            }
            fence_proxy_async();
            __syncwarp();
            const int br = tc.r0 + 2 * bi, bc = tc.c0 + 8 * bj;
            if (lane == 0 && br < p.H && bc < p.W) {
                tma_store_4d(&mO, ob, 0, bc, br, tc.sl);
                bulk_commit();
            }
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ===========================================================================
// host side
// ===========================================================================
constexpr int kSmemPerCta = 226 * 1024;       // dynamic shared memory one CTA may ask for

// Epilogue configuration: one input slot, so that (fixed weights) an epilogue
// CTA fits beside a statistics CTA and starts its loads and first local branch
// while the statistics still run; two B-operand buffers if they fit, else one.
// (Two slots at one CTA per SM measured slower on the PVT-T layer.)
void epi_config(const TcParams &t, bool mlp, int *slots, int *nb, int *smem) {
    *slots = 0;
    for (int b = 2; b >= 1; --b) {
        const int bytes = (int)epi_layout(t.BR, t.BC, t.epi_rows, t.n_mlp, mlp, 1, b).total + 1024;
        if (bytes <= kSmemPerCta && t.slot_cols <= 512) {
            *slots = 1;
            *nb = b;
            *smem = bytes;
            return;
        }
    }
}

}  // namespace

// Epilogue tile: BR x BC blocks of 2 x 8 tokens (BR * BC = 8); fewest tiles.
void tc_tile_shape(int H, int W, int *BR, int *BC) {
    static const int shapes[3][2] = {{4, 2}, {8, 1}, {2, 4}};
    long best = -1;
    for (auto &s : shapes) {
        const long t = (long)((H + 2 * s[0] - 1) / (2 * s[0])) * ((W + 8 * s[1] - 1) / (8 * s[1]));
        if (best < 0 || t < best) {
            best = t;
            *BR = s[0];
            *BC = s[1];
        }
    }
}

// The fused stats kernel needs all of a slice's chunks in one cluster and the
// chunk's K rows resident in shared memory.
bool tc_fused(int chunks, int cluster, int chunk) {
    return chunks == cluster && (chunk + kSub - 1) / kSub <= kFusedMaxSub;
}

cudaError_t launch_tc_stats_partials(const Problem &p, cudaStream_t st, bool with_keysum) {
    Problem q = p;
    q.tc_split = 1;
    q.resident = 0;
    cudaError_t err = with_keysum ? launch_tc(q, st, 0) : cudaSuccess;   // key-sum partials
    return err == cudaSuccess ? launch_tc(q, st, 1) : err;              // [U_1^T ; M^T] cluster partials
}

cudaError_t launch_tc(const Problem &p, cudaStream_t st, int stage) {
    if (p.resident)
        return (stage < 0 || stage == 0) ? launch_tc_resident(p, st) : cudaErrorInvalidValue;
    TcParams t{};
    t.slices = p.slices; t.heads = p.heads; t.H = p.H; t.W = p.W; t.n = p.n; t.T = p.T;
    t.relu = p.relu; t.wmode = p.wmode; t.hidden = p.hidden; t.eps = p.eps; t.alpha = p.alpha;
    t.k_raw = p.k_raw;
    t.untruncated = p.untruncated; t.beta = p.beta;
    for (int k = 0; k < LISA_MAX_T; ++k) t.w[k] = p.w[k];
    t.W1 = p.W1; t.b1 = p.b1; t.W2 = p.W2; t.b2 = p.b2; t.K = p.K;
    t.chunks = p.chunks; t.chunk = p.chunk; t.cl = p.tc_cluster; t.parts = p.chunks / p.tc_cluster;
    tc_tile_shape(p.H, p.W, &t.BR, &t.BC);
    t.tiles_r = (p.H + 2 * t.BR - 1) / (2 * t.BR);
    t.tiles_c = (p.W + 8 * t.BC - 1) / (8 * t.BC);
    t.tiles = p.slices * t.tiles_r * t.tiles_c;
    const bool mlp = p.wmode == LISA_W_MLP;
    t.n_umat = mlp ? p.T - 1 : 1;
    t.epi_rows = 64 * t.n_umat + 16;
    t.n_mlp = mlp ? (p.hidden + 15) / 16 * 16 : 0;
    t.slot_cols = (t.epi_rows + t.n_mlp + 31) / 32 * 32;
    t.s_part = p.s_part; t.part = p.tc_part; t.bepi = p.tc_bepi; t.w1img = p.tc_w1img; t.err = p.err;
    const bool fused = !p.tc_split && tc_fused(p.chunks, p.tc_cluster, p.chunk);
    // stage index of each kernel in this chain (-1: not part of it)
    const int s_keysum = fused ? -1 : 0, s_stats = fused ? 0 : 1, s_recur = fused ? -1 : 2,
              s_epi = fused ? 1 : 3;
    auto run = [&](int s) { return s >= 0 && (stage < 0 || stage == s); };

    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = (unsigned)t.cl;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = st;
    cudaError_t err = cudaSuccess;

    if (run(s_keysum)) {   // first kernel of the split chain: programmatic launch, waits on entry
        cfg.gridDim = dim3((unsigned)(p.slices * p.chunks));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
        if ((err = cudaLaunchKernelEx(&cfg, tc_keysum_kernel, t)) != cudaSuccess) return err;
    }
    if (run(s_stats)) {
        CUtensorMap mq, mk, mv;
        if (!make_map_tokens(&mq, p.Q, p.slices, p.n, kSub) || !make_map_tokens(&mk, p.K, p.slices, p.n, kSub) ||
            !make_map_tokens(&mv, p.V, p.slices, p.n, kSub))
            return cudaErrorInvalidValue;
        cfg.gridDim = dim3((unsigned)(p.slices * p.chunks));
        cfg.blockDim = dim3(128);
        if (fused) {
            const int nsub = (p.chunk + kSub - 1) / kSub;
            int kres = nsub * kSubBytes;
            const int ring = kStages * 2 * kSubBytes;
            if (kres + ring < kFusedWork) kres = kFusedWork - ring;
            const int smem = kres + ring + 1024;
            // the untruncated walk has its own instance (the solve's call costs registers)
            auto kern = p.untruncated ? tc_stats_fused_kernel<true> : tc_stats_fused_kernel<false>;
            if ((err = set_smem(kern, p.untruncated ? 4 : 0, smem)) != cudaSuccess) return err;
            cfg.dynamicSmemBytes = smem;
            cfg.blockDim = dim3(kStatsThreads);
            cfg.attrs = attrs;        // first kernel of the fused chain: waits after its set-up
            cfg.numAttrs = 2;
            if ((err = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, t, kres)) != cudaSuccess) return err;
        } else {
            const int smem = kStages * 3 * kSubBytes + 1024;
            if ((err = set_smem(tc_stats_split_kernel, 1, smem)) != cudaSuccess) return err;
            cfg.dynamicSmemBytes = smem;
            cfg.blockDim = dim3(kStatsThreads);
            cfg.attrs = attrs;
            cfg.numAttrs = 2;
            if ((err = cudaLaunchKernelEx(&cfg, tc_stats_split_kernel, mq, mk, mv, t)) != cudaSuccess) return err;
        }
    }
    if (run(s_recur)) {
        cfg.gridDim = dim3((unsigned)(p.slices * kRecurRowBlocks));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
        if ((err = cudaLaunchKernelEx(&cfg, tc_recur_kernel, t)) != cudaSuccess) return err;
    }
    if (run(s_epi)) {
        CUtensorMap mq, mkh, mvh, mkt, mo;
        const int th = 2 * t.BR, tw = 8 * t.BC;
        if (!make_map_grid(&mq, p.Q, p.slices, p.H, p.W, th, 8) ||
            !make_map_grid(&mkh, p.K, p.slices, p.H, p.W, th + 2, tw + 2) ||
            !make_map_grid(&mvh, p.V, p.slices, p.H, p.W, th + 2, tw + 2) ||
            !make_map_grid(&mkt, p.K, p.slices, p.H, p.W, th, 8) ||
            !make_map_grid(&mo, p.O, p.slices, p.H, p.W, 2, 8))   // one warp's 2 x 8 block
            return cudaErrorInvalidValue;
        int slots = 0, nb = 0, smem = 0;
        epi_config(t, mlp, &slots, &nb, &smem);
        if (slots == 0) return cudaErrorInvalidConfiguration;
        t.epi_nbepi = nb;
        const uint32_t cols = pow2_cols(slots * t.slot_cols);
        const int nctas = sm_count();   // one persistent CTA per SM
        cfg.gridDim = dim3((unsigned)(t.tiles < nctas ? t.tiles : nctas));
        cfg.blockDim = dim3(kEpiThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
        auto launch = [&](auto kern, int slot) {
            cudaError_t e = set_smem(kern, slot, smem);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, kern, mq, mkh, mvh, mkt, mo, t, cols);
        };
        err = mlp ? launch(tc_epilogue_kernel<true, 1, 1>, 2) : launch(tc_epilogue_kernel<false, 1, 1>, 3);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

namespace {
__global__ void wait_selftest_kernel(int *err, long long cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    *err = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    // nothing arrives on the barrier: the wait must give up after `cycles`
    if (!mbar_wait_for(smem_u32(&bar), 0, cycles)) record_error(err, kErrTimeoutLoad);
}
}  // namespace

cudaError_t launch_wait_selftest(int *err, long long cycles, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, cycles);
    return cudaGetLastError();
}

int tc_num_stages(int chunks, int cluster, int chunk) { return tc_fused(chunks, cluster, chunk) ? 2 : 4; }

const char *tc_stage_name(int chunks, int cluster, int chunk, int stage) {
    static const char *const split[4] = {"tc_keysum", "tc_stats", "tc_recur", "tc_epilogue"};
    static const char *const fused[2] = {"tc_stats_fused", "tc_epilogue"};
    if (tc_fused(chunks, cluster, chunk)) return (stage >= 0 && stage < 2) ? fused[stage] : nullptr;
    return (stage >= 0 && stage < 4) ? split[stage] : nullptr;
}

}  // namespace lisa
