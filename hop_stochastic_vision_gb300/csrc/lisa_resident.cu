// lisa_resident.cu -- single-kernel tensor-core forward of the LiSA layer for
// bf16 layers with d_h = d_v = 64 and walk weights shared by all tokens, on
// grids with an even number of rows and a multiple of 8 columns (<= 64).
//
// "note" below is the reading note of "LiSA: Linear Stochastic Attention for
// Long-Range Visual Modeling" (arXiv 2611.04216v2).  Per (batch, head) slice
// the layer needs the key sum s [note §2.2], the statistics U_1 = K^T V and
// M = K^T Q~ [note §2.3, paper Eq. 8], the recurrence U_k = M U_(k-1), the
// global term Q~_i U-bar, and the 3x3 local branch with the alpha mix
// [note §2.4].
//
// One thread-block cluster per slice; its CL CTAs split the slice's
// block-rows (pairs of grid rows) evenly.  Every input byte crosses from L2
// to the SM once, except Q, which the last phase reads a second time:
//
//  phase 1  TMA loads the CTA's K rows (plus the grid row above and below)
//           and keeps them resident, with the first V and Q rows right behind;
//           ReLU in place; partial key sum; bulk copies push it to every CTA
//           of the cluster, which then add the partials in rank order (s).
//  phase 2  V and Q stream through rings of block-rows.  Four warps form
//           Q~ = Q / (Q.s + eps) of each block-row in place (and keep
//           Q.s + eps per token); one thread then issues tcgen05.mma
//           [V | Q~]^T K into a TMEM accumulator ([U_1^T ; M^T] partial).
//           Per 2 x 8 token block a compute warp runs the 3x3 local branch
//           on the legacy mma.sync path (scores Q~ K^T of the 4 x 10 key
//           window rescaled by Q.s + eps, masked softmax, weights times V,
//           with alpha w_0 folded into the weight of the token itself) and
//           parks (1-alpha) l_i + alpha w_0 V_i in TMEM as bf16.
//  phase 3  the cluster sums the accumulators in fixed rank order (each CTA
//           owns 128/CL rows: bulk copies to the owner, a local sum, bulk
//           copies of the reduced rows to everyone), every CTA runs the
//           recurrence U_k^T = U_(k-1)^T M^T (TF32) -- or, for the
//           untruncated walk, the d x d solve (I - beta M) X = U_1 -- and
//           builds the B operand [U-bar^T | s_hi | s_lo] in shared memory,
//           while the first two phase-4 tiles of Q load.
//  phase 4  per 128-token tile (8 blocks): Q is reloaded (L2) and ReLU'd one
//           tile ahead, tcgen05 forms Q [U-bar | s_hi | s_lo] in TMEM, and
//           each warp adds alpha (Q_i U-bar) / (Q_i . s + eps) to its parked
//           blocks and stores them with TMA.
//
// Warps 0-7 run the local branch and phases 3 and 4, warps 8-11 form Q~,
// warp 12 issues the TMA loads of K, Q and the phase-4 tiles, warp 13 the V
// ring refills, warp 14 every tensor-core MMA.  Every wait is bounded: a wait
// that gives up records a bit in the call's error word and the kernel carries
// on along its normal path, so every CTA still drains its bulk stores and
// frees its TMEM.
//
// DRAM traffic equals the algorithmic bytes, yet each CTA walks its
// block-rows one after another with few warps in flight, so the kernel is
// bound by latency, not bandwidth: on the 56 x 56 PVT stage (32 slices) it
// takes 35.3 us at T = 3 where the two-kernel chain (statistics, then the
// epilogue over the whole GPU) takes 31.8 us.  lisa_forward therefore runs
// the chain; this kernel is reached through lisa_forward_resident, a test
// hook.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lisa_internal.h"
#include "lisa_sm100.cuh"
#include "lisa_solve.cuh"
#include "lisa_tc_common.cuh"

namespace lisa {
namespace {

constexpr int kRcCompute = 8;                  // local-branch warps (two per TMEM lane quadrant)
constexpr int kPerQuad = kRcCompute / 4;
constexpr int kRcComputeThreads = 32 * kRcCompute;
constexpr int kRcQt = kRcCompute;              // first of the four warps that form Q~
constexpr int kQtWarps = 4;
constexpr int kRcControl = kRcQt + kQtWarps;   // TMA warp for K, Q and the phase-4 tiles
constexpr int kRcVload = kRcControl + 1;        // TMA warp for the V ring refills
constexpr int kRcMma = kRcVload + 1;            // MMA warp: lane 0 issues every tensor-core MMA
constexpr int kRcThreads = 32 * (kRcMma + 1);
constexpr int kVPairs = 4;                     // V ring: block-row pairs, plus two halo rows
constexpr int kQPairs = 2;                     // Q ring: block-row pairs
constexpr int kNB = 8;                         // ring of per-block-row barriers
constexpr int kMaxCl = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmPart = 0;                // parked local branch: 32 columns per tile
constexpr uint32_t kTmAcc = 256;               // [U_1^T ; M^T] accumulator, 64 columns
constexpr uint32_t kTmProd = 320;              // phase-4 products, two buffers of 80 columns
constexpr uint32_t kTmProdStride = 96;
constexpr int kQtSlots = 3;                    // TMEM ring of Q~ block-rows for the local branch
constexpr uint32_t kTmQt = 416;                // its 3 x 32 columns (phase 2; the second product buffer in phase 4)
constexpr int kBRows = 80;                     // B operand: 64 rows U-bar^T, s_hi, s_lo, 14 zero rows
constexpr uint32_t kTileBytes = 128 * kRow;    // one phase-4 Q tile (8 blocks of 16 tokens)
constexpr uint32_t kBlkBytes = 16 * kRow;      // one 2 x 8 token block
constexpr int kSmemPerCta = 227 * 1024 - 8192; // dynamic shared memory: the SM's 227 KB less the static part

inline uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

struct RcParams {
    int slices, heads, H, W, n, T, relu, R, CL;
    int untruncated;       // U-bar = beta (1-beta) (I - beta M)^-1 U_1 instead of the series
    float eps, beta;
    const float *alpha;
    float w[LISA_MAX_T];
    int *err;
    int nbx;               // blocks per block-row (W / 8)
    uint32_t rb;           // bytes of one grid row (W * 128)
    uint32_t off_ring;     // V ring (4 pairs + 2 halo rows), then the Q ring (2 pairs)
    // phase 3 overlays of the K region
    uint32_t off_part, off_recv, off_full;
    // phase 3 and 4 overlays: recurrence buffers, B operand, the two Q tiles
    uint32_t off_mt, off_ua, off_ub, off_fold, off_b, off_q4[4], off_stage;
};

struct RcBars {
    uint64_t kfull, s_bar, s_ready, acc_full, all_ready, red_bar, full_bar, b_ready, p2_done;
    uint64_t q_full[kQPairs], v_full[kVPairs + 2], v_empty[kVPairs];
    uint64_t qt_ready[kNB], afrag_done[kNB], local_done[kNB], mma_done[kNB];
    uint64_t q4_full[4], q4_relu[4], mma4_full[4], tmem4_empty[2];
};

// Bulk copy of `bytes` from this CTA's shared memory to the shared memory of
// a CTA of the cluster (dst and its mbarrier given as cluster addresses);
// completion is counted in bytes on that mbarrier.
__device__ __forceinline__ void bulk_s2c(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}
// Arrive on an mbarrier of a CTA of the cluster (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kRcComputeThreads) : "memory");   // the compute warps only
}
struct ComputeSync {
    __device__ __forceinline__ void operator()() const { compute_sync(); }
};
__device__ __forceinline__ void tmem_st_frag16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_ld_frag16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp writes lane
// (base lane + t).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, int *err, int bits) {
    if (!mbar_wait(bar, parity)) record_error(err, bits);
}

// Block `blk` of the CTA (block-row-major order) lives in TMEM tile blk / 8 at
// lane position blk % 8 (16 lanes each), so its lanes sit in quadrant
// (blk % 8) / 2.  The compute warps of that quadrant (warp & 3) take its
// blocks in turn.
__device__ __forceinline__ bool owns_block(int blk, int warp) {
    const int pos = blk & 7;
    return (pos >> 1) == (warp & 3) && ((2 * (blk >> 3) + (pos & 1)) % kPerQuad) == (warp >> 2);
}

// One step of the recurrence on the legacy tensor path, TF32 operands:
// Un = U Mt for 64 x 64 matrices (U, Un, fold with row stride kUS, Mt with
// kMS), and fold += wk Un.  Eight warps: warp w computes rows 16 (w % 4) ..
// + 15 and column tiles 4 (w / 4) .. + 3.  The fp32 bits are the operands
// (the tensor core reads their leading 19 bits).
__device__ __forceinline__ void recur_step_tf32(const float *U, const float *Mt, float *Un, float *fold, float wk,
                                                int warp, int lane) {
    const int g = lane >> 2, q4 = lane & 3;
    const int r0 = 16 * (warp & 3) + g, r1 = r0 + 8, nt0 = 4 * (warp >> 2);
    uint32_t a[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int b = 8 * ks + q4;
        a[ks][0] = __float_as_uint(U[r0 * kUS + b]);
        a[ks][1] = __float_as_uint(U[r1 * kUS + b]);
        a[ks][2] = __float_as_uint(U[r0 * kUS + b + 4]);
        a[ks][3] = __float_as_uint(U[r1 * kUS + b + 4]);
    }
#pragma unroll
    for (int nt = nt0; nt < nt0 + 4; ++nt) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int b = 8 * ks + q4;
            mma_tf32_1688(d, a[ks][0], a[ks][1], a[ks][2], a[ks][3], __float_as_uint(Mt[b * kMS + 8 * nt + g]),
                          __float_as_uint(Mt[(b + 4) * kMS + 8 * nt + g]));
        }
        const int c = 8 * nt + 2 * q4;
        Un[r0 * kUS + c] = d[0];
        Un[r0 * kUS + c + 1] = d[1];
        Un[r1 * kUS + c] = d[2];
        Un[r1 * kUS + c + 1] = d[3];
        fold[r0 * kUS + c] = fmaf(wk, d[0], fold[r0 * kUS + c]);
        fold[r0 * kUS + c + 1] = fmaf(wk, d[1], fold[r0 * kUS + c + 1]);
        fold[r1 * kUS + c] = fmaf(wk, d[2], fold[r1 * kUS + c]);
        fold[r1 * kUS + c + 1] = fmaf(wk, d[3], fold[r1 * kUS + c + 1]);
    }
}

__global__ void __launch_bounds__(kRcThreads, 1)
    tc_resident_kernel(const __grid_constant__ CUtensorMap mQr, const __grid_constant__ CUtensorMap mKr,
                       const __grid_constant__ CUtensorMap mVr, const __grid_constant__ CUtensorMap mQb,
                       const __grid_constant__ CUtensorMap mOb, RcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) RcBars bar;
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float s_all[kMaxCl][kD];   // every CTA's partial key sum, rank order
    __shared__ __align__(16) float s_loc[kD];
    __shared__ __align__(16) float s_sh[kD];
    __shared__ float s_red[kRcCompute][kD];
    __shared__ float r_buf[kQtSlots][128];              // Q_i . s + eps of the TMEM ring's tokens

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int CL = p.CL;
    const int sl = blockIdx.x / CL;
    const int rank = (int)cluster_rank();
    const int jb0 = p.R * rank / CL, jb1 = p.R * (rank + 1) / CL, nbr = jb1 - jb0;
    const int top = jb0 > 0 ? 1 : 0, bottom = jb1 < p.R ? 1 : 0;
    const int y_lo = 2 * jb0 - top;                    // first resident K row (grid row)
    const int nrows = 2 * nbr + top + bottom;
    const int W = p.W, nbx = p.nbx, nblk = nbr * nbx, ntiles = (nblk + 7) / 8;
    const uint32_t RB = p.rb;
    const uint32_t base = smem_u32(sm);
    const uint32_t kbase = base;                        // K region at offset 0
    const uint32_t vbase = base + p.off_ring;           // V ring rows 0..9
    const uint32_t qbase = vbase + (2 * kVPairs + 2) * RB;   // Q ring rows 0..3
    // rows of the reduction this CTA owns
    const int own0 = 128 * rank / CL, own1 = 128 * (rank + 1) / CL, own_rows = own1 - own0;
    const int slot_rows = (128 + CL - 1) / CL;          // receive slot per source rank

    if (tid == 0) {
        mbar_init(smem_u32(&bar.kfull), 1);
        mbar_init(smem_u32(&bar.s_bar), 1);
        mbar_init(smem_u32(&bar.s_ready), 1);
        mbar_init(smem_u32(&bar.acc_full), 1);
        mbar_init(smem_u32(&bar.all_ready), (uint32_t)CL);
        mbar_init(smem_u32(&bar.red_bar), 1);
        mbar_init(smem_u32(&bar.full_bar), 1);
        mbar_init(smem_u32(&bar.b_ready), 1);
        mbar_init(smem_u32(&bar.p2_done), kRcCompute);
        for (int i = 0; i < kQPairs; ++i) mbar_init(smem_u32(&bar.q_full[i]), 1);
        for (int i = 0; i < kVPairs + 2; ++i) mbar_init(smem_u32(&bar.v_full[i]), 1);
        // a V pair is read by the blocks of three block-rows (the windows of the block-rows
        // before, at and after it) and by its block-row's statistics MMA
        for (int i = 0; i < kVPairs; ++i) mbar_init(smem_u32(&bar.v_empty[i]), (uint32_t)(3 * nbx + 1));
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&bar.qt_ready[i]), 1);
            mbar_init(smem_u32(&bar.afrag_done[i]), (uint32_t)nbx);
            mbar_init(smem_u32(&bar.local_done[i]), kRcCompute);
            mbar_init(smem_u32(&bar.mma_done[i]), 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(smem_u32(&bar.q4_full[i]), 1);
            mbar_init(smem_u32(&bar.q4_relu[i]), kRcCompute);
            mbar_init(smem_u32(&bar.mma4_full[i]), 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bar.tmem4_empty[i]), kRcCompute);
        fence_mbar_init();
        // the exchange barriers expect their bytes from the start
        mbar_arrive_expect_tx(smem_u32(&bar.s_bar), (uint32_t)CL * kD * 4u);
        mbar_arrive_expect_tx(smem_u32(&bar.red_bar), (uint32_t)(CL * own_rows) * 256u);
        mbar_arrive_expect_tx(smem_u32(&bar.full_bar), (uint32_t)(128 - own_rows) * 256u);
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // every CTA's barriers exist before the first remote copy or arrive
    const uint32_t tmem = tmem_slot;
    // Launched as a programmatic dependent of the preceding kernel: only set-up
    // above; the inputs are read after this wait returns.
    pdl_wait();
    if (blockIdx.x == 0 && tid == 0) *p.err = 0;
    pdl_launch_dependents();

    // ring fills: V pair jj (block-row jj's two rows) and Q pair jj into their slots
    auto load_vpair = [&](int jj) {
        const int slot = jj % kVPairs;
        const uint32_t b = smem_u32(&bar.v_full[slot]);
        mbar_arrive_expect_tx(b, 2u * RB);
        for (int h = 0; h < 2; ++h)
            tma_load_3d(vbase + (uint32_t)(2 * slot + h) * RB, &mVr, 0, (2 * (jb0 + jj) + h) * W, sl, b);
    };
    auto load_qpair = [&](int jj) {
        const int slot = jj % kQPairs;
        const uint32_t b = smem_u32(&bar.q_full[slot]);
        mbar_arrive_expect_tx(b, 2u * RB);
        for (int h = 0; h < 2; ++h)
            tma_load_3d(qbase + (uint32_t)(2 * slot + h) * RB, &mQr, 0, (2 * (jb0 + jj) + h) * W, sl, b);
    };
    if (warp == kRcControl) {
        // =============================== TMA warp: K, Q and phase-4 tiles (lane 0)
        if (lane == 0) {
            mbar_arrive_expect_tx(smem_u32(&bar.kfull), (uint32_t)nrows * RB);
            for (int r = 0; r < nrows; ++r)
                tma_load_3d(kbase + (uint32_t)r * RB, &mKr, 0, (y_lo + r) * W, sl, smem_u32(&bar.kfull));
            // K gates the key sum, s and every Q~: it lands alone first; the rings fill after
            wait_or_flag(smem_u32(&bar.kfull), 0, p.err, kErrTimeoutLoad);
            for (int jj = 0; jj < kQPairs && jj < nbr; ++jj) load_qpair(jj);
            if (top) {
                const uint32_t b = smem_u32(&bar.v_full[kVPairs]);
                mbar_arrive_expect_tx(b, RB);
                tma_load_3d(vbase + (uint32_t)(2 * kVPairs) * RB, &mVr, 0, (2 * jb0 - 1) * W, sl, b);
            }
            for (int jj = 0; jj < kVPairs && jj < nbr; ++jj) load_vpair(jj);
            if (bottom) {
                const uint32_t b = smem_u32(&bar.v_full[kVPairs + 1]);
                mbar_arrive_expect_tx(b, RB);
                tma_load_3d(vbase + (uint32_t)(2 * kVPairs + 1) * RB, &mVr, 0, 2 * jb1 * W, sl, b);
            }
            // every later V and Q row into L2 now, in the order the ring takes them: the
            // slice's DRAM traffic streams at once and the ring refills hit L2
            for (int jj = 1; jj < nbr; ++jj) {
                if (jj >= kQPairs) {
                    tma_prefetch_3d(&mQr, 0, 2 * (jb0 + jj) * W, sl);
                    tma_prefetch_3d(&mQr, 0, (2 * (jb0 + jj) + 1) * W, sl);
                }
                if (jj + 1 < nbr && jj + 1 >= kVPairs) {
                    tma_prefetch_3d(&mVr, 0, 2 * (jb0 + jj + 1) * W, sl);
                    tma_prefetch_3d(&mVr, 0, (2 * (jb0 + jj + 1) + 1) * W, sl);
                }
            }
        }
        __syncwarp();
        // s = the cluster's partial key sums added in rank order, for every warp of the CTA
        wait_or_flag(smem_u32(&bar.s_bar), 0, p.err, kErrTimeoutLoad);
        for (int e = lane; e < kD; e += 32) {
            float v = 0.f;
            for (int r = 0; r < CL; ++r) v += s_all[r][e];
            s_sh[e] = v;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(smem_u32(&bar.s_ready));
            // Q refills (lane 0), in block-row order
            for (int jj = kQPairs; jj < nbr; ++jj) {
                // its slot is free once that block-row's MMA has read Q~
                const int old = jj - kQPairs;
                wait_or_flag(smem_u32(&bar.mma_done[old % kNB]), (uint32_t)(old / kNB) & 1u, p.err, kErrTimeoutMma);
                load_qpair(jj);
            }
            // phase 4 Q tiles, four buffers: tiles 0 and 1 load during phase 3 (their
            // buffers are free once every compute warp is past phase 2 and the last
            // MMA has run), tiles 2 and 3 once phase 3 is done with the reduction
            // buffers, tile t >= 4 once the MMA of tile t - 4 has read its buffer
            wait_or_flag(smem_u32(&bar.p2_done), 0, p.err, kErrTimeoutLoad);
            wait_or_flag(smem_u32(&bar.acc_full), 0, p.err, kErrTimeoutMma);
            for (int t = 0; t < ntiles; ++t) {
                const int buf = t & 3;
                if (t == 2) wait_or_flag(smem_u32(&bar.b_ready), 0, p.err, kErrTimeoutMma);
                if (t >= 4)
                    wait_or_flag(smem_u32(&bar.mma4_full[buf]), (uint32_t)((t - 4) >> 2) & 1u, p.err,
                                 kErrTimeoutMma);
                const int nb = min(8, nblk - 8 * t);
                const uint32_t b = smem_u32(&bar.q4_full[buf]);
                mbar_arrive_expect_tx(b, (uint32_t)nb * kBlkBytes);
                for (int u = 0; u < nb; ++u) {
                    const int blk = 8 * t + u, jj = blk / nbx, bx = blk % nbx;
                    tma_load_4d(base + p.off_q4[buf] + (uint32_t)u * kBlkBytes, &mQb, 0, 8 * bx, 2 * (jb0 + jj), sl, b);
                }
            }
        }
        __syncwarp();
    } else if (warp >= kRcQt && warp < kRcQt + kQtWarps) {
        // =============================== Q~ = Q / (Q.s + eps) per block-row
        // One warp per TMEM lane quadrant, one thread per token.  Block bx of block-row jj
        // sits at lane position (jj nbx + bx) % 8 -- its position in the parked-output
        // tile, where its local-branch warp reads and writes TMEM -- so lane l of quadrant q
        // holds token (l >> 3) & 1, l & 7 of the block at position 2 q + (l >> 4).  Q~ goes
        // back into the Q ring in place (the statistics MMA reads it there) and into a TMEM
        // ring slot in the mma.sync A-fragment order (the local branch reads it there),
        // with Q.s + eps per token in r_buf.
        const int quad = warp & 3;
        const int pos = 2 * quad + (lane >> 4), tr = (lane >> 3) & 1, tc = lane & 7;
        uint8_t *qring = sm + p.off_ring + (2 * kVPairs + 2) * RB;
        const float4 *s4 = reinterpret_cast<const float4 *>(s_sh);
        wait_or_flag(smem_u32(&bar.s_ready), 0, p.err, kErrTimeoutLoad);
        for (int jj = 0; jj < nbr; ++jj) {
            const int slot = jj % kQPairs, ts = jj % kQtSlots;
            wait_or_flag(smem_u32(&bar.q_full[slot]), (uint32_t)(jj / kQPairs) & 1u, p.err, kErrTimeoutLoad);
            if (jj >= kQtSlots) {   // the local branches of block-row jj - kQtSlots have read the slot
                const int old = jj - kQtSlots;
                wait_or_flag(smem_u32(&bar.afrag_done[old % kNB]), (uint32_t)(old / kNB) & 1u, p.err,
                             kErrTimeoutMma);
            }
            tc_fence_after();
            const int bx = ((pos - jj * nbx) % 8 + 8) % 8;
            const bool act = bx < nbx;
            const int tok = tr * W + 8 * (act ? bx : 0) + tc;   // token of the block-row
            const uint32_t qt = (uint32_t)(2 * slot * W + tok);
            uint4 q[8];
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                q[c] = *reinterpret_cast<uint4 *>(qring + sw128_offset(qt, c));
                if (p.relu) q[c] = relu4(q[c]);
                const float4 sa = s4[2 * c], sb = s4[2 * c + 1];
                float &acc = part[c & 3];
                acc = fmaf(bf16_lo(q[c].x), sa.x, acc);
                acc = fmaf(bf16_hi(q[c].x), sa.y, acc);
                acc = fmaf(bf16_lo(q[c].y), sa.z, acc);
                acc = fmaf(bf16_hi(q[c].y), sa.w, acc);
                acc = fmaf(bf16_lo(q[c].z), sb.x, acc);
                acc = fmaf(bf16_hi(q[c].z), sb.y, acc);
                acc = fmaf(bf16_lo(q[c].w), sb.z, acc);
                acc = fmaf(bf16_hi(q[c].w), sb.w, acc);
            }
            const float rr = ((part[0] + part[1]) + (part[2] + part[3])) + p.eps, r = 1.f / rr;
            uint32_t pk[32];   // feature pairs (2 m, 2 m + 1), m = 4 c + word
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t w4[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) pk[4 * c + e] = pack_bf16(bf16_lo(w4[e]) * r, bf16_hi(w4[e]) * r);
            }
            if (act) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(qring + sw128_offset(qt, c)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                r_buf[ts][tok] = rr;
            }
            // TMEM columns of a k-step (8 pairs): column 2 u + e holds pair u + 4 e, so that a
            // 16x256b load returns (a0, a2, a1, a3) of the mma.sync A fragment
            uint32_t col[32];
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) col[cc] = pk[8 * (cc >> 3) + ((cc & 7) >> 1) + 4 * (cc & 1)];
            tmem_st32(tmem + kTmQt + 32u * (uint32_t)ts + ((uint32_t)(32 * quad) << 16), col);
            tc_wait_st();
            fence_proxy_async();   // Q~ (generic writes) before the tensor core reads it
            tc_fence_before();
            asm volatile("bar.sync 2, %0;" ::"n"(32 * kQtWarps) : "memory");
            if (warp == kRcQt && lane == 0) mbar_arrive(smem_u32(&bar.qt_ready[jj % kNB]));
        }
    } else if (warp == kRcVload) {
        // =============================== TMA warp: V ring refills (lane 0)
        if (lane == 0) {
            // V refills in a warp of their own, so that their waits never hold up a Q refill: V pair
            // nxt reuses the slot of block-row old = nxt - kVPairs, free once block-row
            // old + 1's local branch (its last reader) and block-row old's MMA are done
            for (int nxt = kVPairs; nxt < nbr; ++nxt) {
                const int old = nxt - kVPairs;   // the slot's last use: V pair old, free once its readers are done
                wait_or_flag(smem_u32(&bar.v_empty[old % kVPairs]), (uint32_t)(old / kVPairs) & 1u, p.err,
                             kErrTimeoutMma);
                load_vpair(nxt);
            }
        }
        __syncwarp();
    } else if (warp == kRcMma) {
        // =============================== tensor-core issue
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_bf16(128, 64, true, true);
            for (int jj = 0; jj < nbr; ++jj) {
                wait_or_flag(smem_u32(&bar.qt_ready[jj % kNB]), (uint32_t)(jj / kNB) & 1u, p.err, kErrTimeoutLoad);
                wait_or_flag(smem_u32(&bar.v_full[jj % kVPairs]), (uint32_t)(jj / kVPairs) & 1u, p.err, kErrTimeoutLoad);
                tc_fence_after();
                const uint32_t va = vbase + (uint32_t)(2 * (jj % kVPairs)) * RB;
                const uint32_t qa = qbase + (uint32_t)(2 * (jj % kQPairs)) * RB;
                const uint32_t ka = kbase + (uint32_t)(2 * jj + top) * RB;
                for (int ks = 0; ks < nbx; ++ks) {   // 2W tokens = W / 8 steps of 16
                    const uint64_t ad = make_desc_sw128(va + ks * 2048, qa - va, 1024);
                    const uint64_t bd = make_desc_sw128(ka + ks * 2048, 1024, 1024);
                    tc_mma(tmem + kTmAcc, ad, bd, idesc, (jj | ks) != 0);
                }
                tc_commit(smem_u32(&bar.mma_done[jj % kNB]));
                tc_commit(smem_u32(&bar.v_empty[jj % kVPairs]));   // the MMA's read of V pair jj
            }
            tc_commit(smem_u32(&bar.acc_full));
            // phase 4: Q [U-bar | s_hi | s_lo] per tile
            wait_or_flag(smem_u32(&bar.b_ready), 0, p.err, kErrTimeoutMma);
            constexpr uint32_t idesc4 = make_idesc_bf16(128, kBRows, false, false);
            const uint32_t ba = base + p.off_b;
            for (int t = 0; t < ntiles; ++t) {
                const int qb = t & 3, tb = t & 1;   // Q buffer, TMEM product buffer
                wait_or_flag(smem_u32(&bar.q4_relu[qb]), (uint32_t)(t >> 2) & 1u, p.err, kErrTimeoutLoad);
                if (t >= 2)
                    wait_or_flag(smem_u32(&bar.tmem4_empty[tb]), (uint32_t)((t - 2) >> 1) & 1u, p.err,
                                 kErrTimeoutMma);
                tc_fence_after();
                const uint32_t qa = base + p.off_q4[qb];
                const uint32_t d = tmem + kTmProd + (uint32_t)tb * kTmProdStride;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc_mma(d, make_desc_sw128(qa + ks * 32, 16, 1024), make_desc_sw128(ba + ks * 32, 16, 1024), idesc4,
                           ks > 0);
                tc_commit(smem_u32(&bar.mma4_full[qb]));
            }
        }
        __syncwarp();
    } else {
        // =============================== compute warps
        // ---- phase 1: ReLU of the resident K in place, partial key sum over the own rows
        wait_or_flag(smem_u32(&bar.kfull), 0, p.err, kErrTimeoutLoad);
        {
            constexpr int kLanes = kRcComputeThreads / 8;   // token lanes x 8 feature chunks
            const int cg = tid & 7, jl = tid >> 3;
            const int own_lo = top * W, own_hi = (top + 2 * nbr) * W, all = nrows * W;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            uint8_t *kres = sm;
            for (int t0 = jl; t0 < all; t0 += 4 * kLanes) {   // four tokens per thread in flight
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = t0 + kLanes * u;
                    v[u] = t < all ? *reinterpret_cast<const uint4 *>(kres + sw128_offset(t, cg)) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = t0 + kLanes * u;
                    if (t >= all) continue;
                    if (p.relu) {
                        v[u] = relu4(v[u]);
                        *reinterpret_cast<uint4 *>(kres + sw128_offset(t, cg)) = v[u];
                    }
                    if (t >= own_lo && t < own_hi) {
                        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[2 * e] += bf16_lo(w4[e]);
                            acc[2 * e + 1] += bf16_hi(w4[e]);
                        }
                    }
                }
            }
            // lanes l, l + 8, l + 16, l + 24 hold the same feature chunk
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
                acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
            }
            if (lane < 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) s_red[warp][cg * 8 + e] = acc[e];
        }
        fence_proxy_async();   // the ReLU'd K (generic writes) before the tensor core reads it
        compute_sync();
        if (tid < kD) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kRcCompute; ++w) s += s_red[w][tid];
            s_loc[tid] = s;
        }
        fence_proxy_async();   // s_loc (generic writes) before the bulk copies read it
        compute_sync();
        if (tid == 0)
            for (int r = 0; r < CL; ++r)
                bulk_s2c(map_rank(smem_u32(&s_all[rank][0]), (uint32_t)r), smem_u32(s_loc), kD * 4u,
                         map_rank(smem_u32(&bar.s_bar), (uint32_t)r));
        // ---- phase 2: per block: the local branch on Q~ (scores rescaled by Q.s + eps), parked in TMEM
        const int g = lane >> 2, q4 = lane & 3;
        uint32_t win_mask = 0, ctr_mask = 0;   // bit j*4+e: key in the query's 3x3 window / the token itself
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
        const float c2 = 1.4426950408889634f * 0.125f;        // log2(e) / sqrt(64)
        const float alpha = p.alpha[sl % p.heads];
        const float self = alpha * p.w[0];
        // ring row of V grid row y (clamped into the resident range: such keys are masked)
        auto vrow = [&](int y) -> int {
            if (y < 2 * jb0) return top ? 2 * kVPairs : 0;
            if (y >= 2 * jb1) return bottom ? 2 * kVPairs + 1 : 2 * ((nbr - 1) % kVPairs) + 1;
            const int r = y - 2 * jb0;
            return 2 * ((r >> 1) % kVPairs) + (r & 1);
        };
        for (int jj = 0; jj < nbr; ++jj) {
            wait_or_flag(smem_u32(&bar.qt_ready[jj % kNB]), (uint32_t)(jj / kNB) & 1u, p.err, kErrTimeoutLoad);
            if (jj == 0) {
                if (top) wait_or_flag(smem_u32(&bar.v_full[kVPairs]), 0, p.err, kErrTimeoutLoad);
            } else {
                wait_or_flag(smem_u32(&bar.v_full[(jj - 1) % kVPairs]), (uint32_t)((jj - 1) / kVPairs) & 1u, p.err,
                             kErrTimeoutLoad);
            }
            wait_or_flag(smem_u32(&bar.v_full[jj % kVPairs]), (uint32_t)(jj / kVPairs) & 1u, p.err, kErrTimeoutLoad);
            if (jj + 1 < nbr)
                wait_or_flag(smem_u32(&bar.v_full[(jj + 1) % kVPairs]), (uint32_t)((jj + 1) / kVPairs) & 1u, p.err,
                             kErrTimeoutLoad);
            else if (bottom)
                wait_or_flag(smem_u32(&bar.v_full[kVPairs + 1]), 0, p.err, kErrTimeoutLoad);
            const int yb = 2 * (jb0 + jj);                         // first grid row of the block-row
            for (int bx = 0; bx < nbx; ++bx) {
                const int blk = jj * nbx + bx;
                if (!owns_block(blk, warp)) continue;
                const int tile = blk >> 3, pos = blk & 7;
                const uint32_t lane_base = (uint32_t)(16 * pos) << 16;
                const int x0 = 8 * bx;
                // -- A fragments of the block's 16 queries: Q~ (non-negative) from the TMEM
                // ring, and the two row scales of this lane, q_i . k_j = (Q_i . s + eps) (Q~_i . k_j)
                const int ts = jj % kQtSlots;
                uint32_t a[4][4];
                {
                    uint32_t rq[16];
                    tc_fence_after();
                    tmem_ld_frag16_nowait(tmem + kTmQt + 32u * (uint32_t)ts + lane_base, rq);
                    tc_wait_ld();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        a[ks][0] = rq[4 * ks];
                        a[ks][1] = rq[4 * ks + 2];
                        a[ks][2] = rq[4 * ks + 1];
                        a[ks][3] = rq[4 * ks + 3];
                    }
                }
                const float c2r[2] = {c2 * r_buf[ts][x0 + g], c2 * r_buf[ts][W + x0 + g]};
                tc_fence_before();
                __syncwarp();   // every lane holds its fragments and scales: the TMEM slot may be refilled
                if (lane == 0) mbar_arrive(smem_u32(&bar.afrag_done[jj % kNB]));

                // -- scores against the 4 x 10 key window (resident K, already ReLU'd)
                float sc[5][4];
#pragma unroll
                for (int j = 0; j < 5; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                {
                    uint32_t ktok[3];
#pragma unroll
                    for (int pr = 0; pr < 3; ++pr) {
                        int kk = 8 * (2 * pr + (lane >> 4)) + (lane & 7);
                        kk = kk < 40 ? kk : 0;
                        int ry = yb - 1 + kk / 10 - y_lo;
                        ry = min(max(ry, 0), nrows - 1);
                        const int x = min(max(x0 - 1 + kk % 10, 0), W - 1);
                        ktok[pr] = (uint32_t)(ry * W + x);
                    }
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                        for (int pr = 0; pr < 3; ++pr) {
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(kbase + sw128_offset(ktok[pr], 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
                            mma_bf16_16816(sc[2 * pr], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
                            if (pr < 2) mma_bf16_16816(sc[2 * pr + 1], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b2, b3);
                        }
                }
                // -- masked softmax; the token's own weight also carries alpha w_0
                {
                    const int gr0 = yb - 1, gc0 = x0 - 1;   // grid position of window key (0, 0)
                    uint32_t mask = win_mask;
                    if (gr0 < 0 || gr0 + 3 >= p.H || gc0 < 0 || gc0 + 9 >= W) {
#pragma unroll
                        for (int j = 0; j < 5; ++j)
#pragma unroll
                            for (int b = 0; b < 2; ++b) {
                                const int kappa = 8 * j + 2 * q4 + b;
                                const int gr = gr0 + kappa / 10, gc = gc0 + kappa % 10;
                                if (gr < 0 || gr >= p.H || gc < 0 || gc >= W) mask &= ~(0x5u << (j * 4 + b));
                            }
                    }
#pragma unroll
                    for (int j = 0; j < 5; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[j][e] = ((mask >> (j * 4 + e)) & 1u) ? sc[j][e] * c2r[e >> 1] : -INFINITY;
                }
                float mx[2], sum[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float m0 = fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), m1 = fmaxf(sc[1][2 * h], sc[1][2 * h + 1]);
                    const float m2 = fmaxf(sc[2][2 * h], sc[2][2 * h + 1]), m3 = fmaxf(sc[3][2 * h], sc[3][2 * h + 1]);
                    const float m4 = fmaxf(sc[4][2 * h], sc[4][2 * h + 1]);
                    mx[h] = fmaxf(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)), m4);
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
                    const float s0 = sc[0][2 * h] + sc[0][2 * h + 1], s1 = sc[1][2 * h] + sc[1][2 * h + 1];
                    const float s2 = sc[2][2 * h] + sc[2][2 * h + 1], s3 = sc[3][2 * h] + sc[3][2 * h + 1];
                    const float s4 = sc[4][2 * h] + sc[4][2 * h + 1];
                    sum[h] = ((s0 + s1) + (s2 + s3)) + s4;
                    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
                    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
                }
                float scale[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) scale[h] = sum[h] > 0.f ? __fdividef(1.f - alpha, sum[h]) : 0.f;
#pragma unroll
                for (int j = 0; j < 5; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[j][e] = fmaf(sc[j][e], scale[e >> 1], ((ctr_mask >> (j * 4 + e)) & 1u) ? self : 0.f);
                // -- weights times the V window (V ring)
                float lacc[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) lacc[nt][0] = lacc[nt][1] = lacc[nt][2] = lacc[nt][3] = 0.f;
                {
                    uint32_t vtok[3];
#pragma unroll
                    for (int ks = 0; ks < 3; ++ks) {
                        int kv = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
                        kv = kv < 40 ? kv : 0;
                        const int x = min(max(x0 - 1 + kv % 10, 0), W - 1);
                        vtok[ks] = (uint32_t)(vrow(yb - 1 + kv / 10) * W + x);
                    }
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
                            ldsm_x4_t(vbase + sw128_offset(vtok[ks], 2 * np + (lane >> 4)), b0, b1, b2, b3);
                            mma_bf16_16816(lacc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
                            mma_bf16_16816(lacc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
                        }
                    }
                }
                // -- the V window has been read: release its pairs (jj - 1, jj, jj + 1); the first
                // and the last block-row stand in for the missing neighbour of the edge pairs, so
                // every pair sees 3 nbx block arrivals
                __syncwarp();
                if (lane == 0) {
                    for (int pp = jj - 1; pp <= jj + 1; ++pp) {
                        const int q = pp < 0 ? 0 : (pp >= nbr ? nbr - 1 : pp);
                        mbar_arrive(smem_u32(&bar.v_empty[q % kVPairs]));
                    }
                }
                // -- park (1-alpha) l + alpha w_0 V in TMEM as bf16 pairs (fragment layout)
                {
                    uint32_t r[16];
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        r[4 * rr + 0] = pack_bf16(lacc[2 * rr][0], lacc[2 * rr][1]);
                        r[4 * rr + 1] = pack_bf16(lacc[2 * rr + 1][0], lacc[2 * rr + 1][1]);
                        r[4 * rr + 2] = pack_bf16(lacc[2 * rr][2], lacc[2 * rr][3]);
                        r[4 * rr + 3] = pack_bf16(lacc[2 * rr + 1][2], lacc[2 * rr + 1][3]);
                    }
                    tmem_st_frag16(tmem + kTmPart + 32u * (uint32_t)tile + lane_base, r);
                    tc_wait_st();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.local_done[jj % kNB]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar.p2_done));

        // ---- phase 3: cluster reduction of [U_1^T ; M^T] in fixed rank order, recurrence
        compute_sync();   // every compute warp is past its last read of the resident K
        wait_or_flag(smem_u32(&bar.acc_full), 0, p.err, kErrTimeoutMma);
        tc_fence_after();
        // this CTA's K region is no longer read: every rank may copy into it
        if (warp == 4 && lane < CL) mbar_arrive_cluster(map_rank(smem_u32(&bar.all_ready), (uint32_t)lane));
        float *part = reinterpret_cast<float *>(sm + p.off_part);    // [128][64]
        float *recv = reinterpret_cast<float *>(sm + p.off_recv);    // [CL][slot_rows][64]
        float *full = reinterpret_cast<float *>(sm + p.off_full);    // [128][64]
        if (warp < 4) {
            const int row = 32 * warp + lane;
            uint32_t r[4][16];
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) tmem_ld16(tmem + kTmAcc + ((uint32_t)(32 * warp) << 16) + 16 * cb, r[cb]);
            tc_wait_ld();
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float4 *dst = reinterpret_cast<float4 *>(part + row * 64 + 16 * cb);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dst[k] = make_float4(__uint_as_float(r[cb][4 * k]), __uint_as_float(r[cb][4 * k + 1]),
                                         __uint_as_float(r[cb][4 * k + 2]), __uint_as_float(r[cb][4 * k + 3]));
            }
        }
        fence_proxy_async();
        compute_sync();
        wait_or_flag(smem_u32(&bar.all_ready), 0, p.err, kErrTimeoutLoad);
        if (warp == 0 && lane < CL) {
            const int r = lane, r0 = 128 * r / CL, r1 = 128 * (r + 1) / CL;
            bulk_s2c(map_rank(base + p.off_recv + (uint32_t)(rank * slot_rows) * 256u, (uint32_t)r),
                     base + p.off_part + (uint32_t)r0 * 256u, (uint32_t)(r1 - r0) * 256u,
                     map_rank(smem_u32(&bar.red_bar), (uint32_t)r));
        }
        wait_or_flag(smem_u32(&bar.red_bar), 0, p.err, kErrTimeoutLoad);
        for (int item = tid; item < own_rows * 16; item += kRcComputeThreads) {
            const int i = item >> 4, f = item & 15;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < CL; ++q) {
                const float4 v = reinterpret_cast<const float4 *>(recv + (q * slot_rows + i) * 64)[f];
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            reinterpret_cast<float4 *>(full + (own0 + i) * 64)[f] = acc;
        }
        fence_proxy_async();
        compute_sync();
        if (warp == 0 && lane < CL && lane != rank)
            bulk_s2c(map_rank(base + p.off_full + (uint32_t)own0 * 256u, (uint32_t)lane),
                     base + p.off_full + (uint32_t)own0 * 256u, (uint32_t)own_rows * 256u,
                     map_rank(smem_u32(&bar.full_bar), (uint32_t)lane));
        wait_or_flag(smem_u32(&bar.full_bar), 0, p.err, kErrTimeoutLoad);
        // U_1^T (rows 0..63) and M^T (rows 64..127) into the recurrence's padded layouts
        float *Mt = reinterpret_cast<float *>(sm + p.off_mt);
        float *Ua = reinterpret_cast<float *>(sm + p.off_ua);
        float *Ub = reinterpret_cast<float *>(sm + p.off_ub);
        float *Fold = reinterpret_cast<float *>(sm + p.off_fold);
        const float w1 = p.T > 1 ? p.w[1] : 0.f;   // T = 1: no hop terms, the fold stays zero
        for (int item = tid; item < 64 * 16; item += kRcComputeThreads) {
            const int i = item >> 4, f = item & 15;
            const float4 u = reinterpret_cast<const float4 *>(full + i * 64)[f];
            float4 m = reinterpret_cast<const float4 *>(full + (64 + i) * 64)[f];
            if (p.untruncated) {   // A = I - beta M in place of M^T: element (a, b) at Mt[b][a]
                const int a = 4 * f;
                m = make_float4((a == i ? 1.f : 0.f) - p.beta * m.x, (a + 1 == i ? 1.f : 0.f) - p.beta * m.y,
                                (a + 2 == i ? 1.f : 0.f) - p.beta * m.z, (a + 3 == i ? 1.f : 0.f) - p.beta * m.w);
            }
            reinterpret_cast<float4 *>(Ua + i * kUS)[f] = u;
            reinterpret_cast<float4 *>(Mt + i * kMS)[f] = m;
            reinterpret_cast<float4 *>(Fold + i * kUS)[f] = make_float4(w1 * u.x, w1 * u.y, w1 * u.z, w1 * u.w);
        }
        compute_sync();
        if (p.untruncated) {
            // the untruncated walk: X = (I - beta M)^-1 U_1 replaces the series,
            // its rows (columns of X) overwrite U_1^T; U-bar = beta (1-beta) X
            solve_walk_system<kRcCompute, (128 + kRcCompute - 1) / kRcCompute>(
                Mt, kMS, Ua, kUS, 64, 64, &s_red[0][0], tid, ComputeSync());
            for (int item = tid; item < 64 * 16; item += kRcComputeThreads) {
                const int i = item >> 4, f = item & 15;
                const float4 x = reinterpret_cast<const float4 *>(Ua + i * kUS)[f];
                reinterpret_cast<float4 *>(Fold + i * kUS)[f] = make_float4(w1 * x.x, w1 * x.y, w1 * x.z, w1 * x.w);
            }
            compute_sync();
        }
        {
            float *ua = Ua, *ub = Ub;
            for (int k = 2; k < p.T; ++k) {
                if (warp < 8) recur_step_tf32(ua, Mt, ub, Fold, p.w[k], warp, lane);
                compute_sync();
                float *tmp = ua;
                ua = ub;
                ub = tmp;
            }
        }
        {
            uint8_t *img = sm + p.off_b;
            for (int item = tid; item < 64 * 8; item += kRcComputeThreads) {
                const int i = item >> 3, chunk = item & 7;
                put_row_bf16(img, i, Fold + i * kUS + chunk * 8, chunk);
            }
            wait_or_flag(smem_u32(&bar.s_ready), 0, p.err, kErrTimeoutLoad);   // s, written by the producer warp
            put_s_rows(img, 64, s_sh, tid);
        }
        fence_proxy_async();
        compute_sync();
        if (tid == 0) mbar_arrive(smem_u32(&bar.b_ready));

        // ---- phase 4: global term, mix with the parked local branch, store
        // ReLU of a tile's Q rows of this warp's blocks, then the hand-off to the MMA thread
        auto relu_tile = [&](int t) {
            const int buf = t & 3;
            wait_or_flag(smem_u32(&bar.q4_full[buf]), (uint32_t)(t >> 2) & 1u, p.err, kErrTimeoutLoad);
            if (p.relu) {
                for (int e = 0; e < 2; ++e) {
                    const int pos = 2 * (warp & 3) + e, blk = 8 * t + pos;
                    if (blk >= nblk || !owns_block(blk, warp)) continue;
                    uint4 *v = reinterpret_cast<uint4 *>(sm + p.off_q4[buf] + pos * kBlkBytes);
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[lane + 32 * u] = relu4(v[lane + 32 * u]);
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.q4_relu[buf]));
        };
        // the MMA of tile t + 1 runs while tile t is mixed: ReLU two tiles ahead
        if (ntiles > 0) relu_tile(0);
        if (ntiles > 1) relu_tile(1);
        const uint32_t stage = base + p.off_stage + (uint32_t)warp * kBlkBytes;   // this warp's output block
        for (int t = 0; t < ntiles; ++t) {
            const int qb = t & 3, tb = t & 1;
            if (t + 2 < ntiles) relu_tile(t + 2);
            wait_or_flag(smem_u32(&bar.mma4_full[qb]), (uint32_t)(t >> 2) & 1u, p.err, kErrTimeoutMma);
            tc_fence_after();
            for (int e = 0; e < 2; ++e) {
                const int pos = 2 * (warp & 3) + e, blk = 8 * t + pos;
                if (blk >= nblk || !owns_block(blk, warp)) continue;
                const uint32_t tl = tmem + ((uint32_t)(16 * pos) << 16);
                uint32_t ru[32], rs[4], rp[16];
                tmem_ld_frag8_nowait(tl + kTmProd + (uint32_t)tb * kTmProdStride, ru);
                tmem_ld_frag_nowait(tl + kTmProd + (uint32_t)tb * kTmProdStride + 64, rs);
                tmem_ld_frag16_nowait(tl + kTmPart + 32u * (uint32_t)t, rp);
                tc_wait_ld();
                const int src = lane & ~3;
                const float d0 = __shfl_sync(0xffffffffu, __uint_as_float(rs[0]) + __uint_as_float(rs[1]), src);
                const float d1 = __shfl_sync(0xffffffffu, __uint_as_float(rs[2]) + __uint_as_float(rs[3]), src);
                const float arq[2] = {__fdividef(alpha, d0 + p.eps), __fdividef(alpha, d1 + p.eps)};
                if (lane == 0) bulk_wait_read<0>();   // the previous store has read the staging buffer
                __syncwarp();
#pragma unroll
                for (int nt0 = 0; nt0 < 8; nt0 += 2) {
                    uint32_t r[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int nt = nt0 + (m >> 1), h = m & 1;
                        // parked pair of n-tile nt, row g (h = 0) or g + 8 (h = 1)
                        const uint32_t pk = rp[4 * (nt >> 1) + 2 * h + (nt & 1)];
                        r[m] = pack_bf16(fmaf(arq[h], __uint_as_float(ru[4 * nt + 2 * h]), bf16_lo(pk)),
                                         fmaf(arq[h], __uint_as_float(ru[4 * nt + 2 * h + 1]), bf16_hi(pk)));
                    }
                    const uint32_t mrow = (uint32_t)(lane & 7), mm = (uint32_t)(lane >> 3);
                    stsm_x4(stage + (8u * (mm & 1u) + mrow) * kRow + ((((uint32_t)nt0 + (mm >> 1)) ^ mrow) << 4), r[0],
                            r[1], r[2], r[3]);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    const int jj = blk / nbx, bx = blk % nbx;
                    tma_store_4d(&mOb, stage, 0, 8 * bx, 2 * (jb0 + jj), sl);
                    bulk_commit();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar.tmem4_empty[tb]));
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while a peer may still copy into its shared memory
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

struct RcPlan {
    int CL, R, nbr_max, smem;
    RcParams layout;
};

bool rc_plan(int slices, int H, int W, int *cl_out, RcPlan *out) {
    if (H < 2 || H % 2 != 0 || W < 8 || W % 8 != 0 || W > 64) return false;
    const int R = H / 2;
    const int sms = sm_count();
    int CL = sms / (slices > 0 ? slices : 1);
    if (CL > kMaxCl) CL = kMaxCl;
    if (CL > R) CL = R;
    if (CL < 1) CL = 1;
    const int nbr_max = (R + CL - 1) / CL;
    const int nblk = nbr_max * (W / 8);
    if ((nblk + 7) / 8 * 32 > (int)kTmAcc) return false;   // parked tiles must fit below the accumulator
    const uint32_t rb = (uint32_t)W * kRow;
    const uint32_t krows = (uint32_t)(2 * nbr_max + 2) * rb;
    // K region: the resident rows; later the reduction buffers and one phase-4 Q tile
    const uint32_t slot_rows = (uint32_t)(128 + CL - 1) / (uint32_t)CL;
    const uint32_t red = align1k(128u * 256u + (uint32_t)CL * slot_rows * 256u + 128u * 256u);
    const uint32_t kneed = red + kTileBytes;
    const uint32_t kreg = align1k(krows > kneed ? krows : kneed);
    // ring region: V ring (10 rows) and Q ring (4 rows); later the recurrence
    // buffers, the B operand and the other phase-4 Q tile
    const uint32_t rings = (uint32_t)(2 * kVPairs + 2 + 2 * kQPairs) * rb;
    const uint32_t mt = 64u * kMS * 4u, us = 64u * kUS * 4u;
    const uint32_t b_off = align1k(mt + 3u * us);
    const uint32_t q4_off = align1k(b_off + (uint32_t)kBRows * kRow);
    const uint32_t rneed = q4_off + kTileBytes;
    const uint32_t rreg = align1k(rings > rneed ? rings : rneed);
    const int smem = (int)(kreg + rreg + 1024);
    if (smem > kSmemPerCta) return false;
    if (cl_out) *cl_out = CL;
    if (out) {
        out->CL = CL;
        out->R = R;
        out->nbr_max = nbr_max;
        out->smem = smem;
        RcParams &L = out->layout;
        L.rb = rb;
        L.off_ring = kreg;
        L.off_part = 0;
        L.off_recv = 128u * 256u;
        L.off_full = L.off_recv + (uint32_t)CL * slot_rows * 256u;
        L.off_q4[1] = red;            // K region, past the reduction buffers
        L.off_q4[2] = 32u * 1024u;    // K region over the reduction buffers: loaded after phase 3
        L.off_q4[3] = 48u * 1024u;
        L.off_stage = 0;              // K region over the stats read-out (phase 4 only)
        L.off_mt = kreg;
        L.off_ua = kreg + mt;
        L.off_ub = L.off_ua + us;
        L.off_fold = L.off_ub + us;
        L.off_b = kreg + b_off;
        L.off_q4[0] = kreg + q4_off;  // ring region, past the B operand
    }
    return true;
}

}  // namespace

bool tc_resident_applies(int slices, int H, int W, int D, int dtype, int wmode, int untruncated, int relu) {
    (void)untruncated;   // the untruncated walk runs here too (its d x d solve in phase 3)
    if (D != 64 || dtype != LISA_BF16 || wmode != LISA_W_FIXED || relu < 0 || relu > 1) return false;
    return rc_plan(slices, H, W, nullptr, nullptr);
}

cudaError_t launch_tc_resident(const Problem &p, cudaStream_t st) {
    RcPlan pl{};
    if (!rc_plan(p.slices, p.H, p.W, nullptr, &pl)) return cudaErrorInvalidConfiguration;
    RcParams t = pl.layout;
    t.slices = p.slices; t.heads = p.heads; t.H = p.H; t.W = p.W; t.n = p.n; t.T = p.T;
    t.relu = p.relu; t.R = pl.R; t.CL = pl.CL; t.eps = p.eps; t.alpha = p.alpha; t.err = p.err;
    t.untruncated = p.untruncated; t.beta = p.beta;
    for (int k = 0; k < LISA_MAX_T; ++k) t.w[k] = p.w[k];
    t.nbx = p.W / 8;
    CUtensorMap mq, mk, mv, mqb, mob;
    if (!make_map_tokens(&mq, p.Q, p.slices, p.n, p.W) || !make_map_tokens(&mk, p.K, p.slices, p.n, p.W) ||
        !make_map_tokens(&mv, p.V, p.slices, p.n, p.W) || !make_map_grid(&mqb, p.Q, p.slices, p.H, p.W, 2, 8) ||
        !make_map_grid(&mob, p.O, p.slices, p.H, p.W, 2, 8))
        return cudaErrorInvalidValue;
    cudaError_t err = set_smem(tc_resident_kernel, 0, pl.smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = (unsigned)pl.CL;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = st;
    cfg.gridDim = dim3((unsigned)(p.slices * pl.CL));
    cfg.blockDim = dim3(kRcThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    if ((err = cudaLaunchKernelEx(&cfg, tc_resident_kernel, mq, mk, mv, mqb, mob, t)) != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace lisa
