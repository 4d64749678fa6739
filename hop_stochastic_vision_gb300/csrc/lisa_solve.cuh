// lisa_solve.cuh -- the d x d system of the untruncated geometric walk,
// solved by one thread block in shared memory.
//
// Without truncation the walk weights are (1-beta) beta^k for every k >= 0
// and the global branch is (1-beta) (I - beta S)^-1 V ("LiSA: Linear
// Stochastic Attention for Long-Range Visual Modeling", reading note, §2.3:
// the closing remark on the geometric series).  With S = Q~ K^T the
// push-through identity (I - beta Q~ K^T)^-1 = I + beta Q~ (I - beta M)^-1 K^T,
// M = K^T Q~, moves the inverse to d x d: the hop terms are
// beta (1-beta) Q~ X with (I - beta M) X = U_1 = K^T V.
#pragma once

namespace lisa {

// Solves (I - beta M) X = R in place: on return A is spent and R holds X.
//
// A = I - beta M is a nonsingular M-matrix: M = K^T Q~ is entrywise
// non-negative (the feature-mapped Q and K are), and its spectral radius is
// that of the row-substochastic S = Q~ K^T, below 1.  Gaussian elimination
// on such a matrix needs no pivoting (every pivot stays positive), so this
// is Gauss-Jordan without row exchanges or row scaling: step p subtracts
// (A_ap / A_pp) times row p from every other row a, on the columns of A still
// live (> p) and on every column of R; A ends diagonal and X_a = R_a / A_aa.
//
// Layout: column b of A (already I - beta M) starts at A + b * sb and column
// e of R at R + e * re, rows contiguous within a column, all in shared
// memory.  The block holds [A | R] in registers: lane l of warp w owns rows
// l and l + 32 of the columns w, w + kW, w + 2 kW, ... (slot k holds column
// w + k kW; kC slots cover D + m <= kC kW columns).  Step p reads row p of
// its own columns from lane p mod 32 by a shuffle and the pivot column from
// shared memory, where its owner published it (the pivot entry itself
// replaced by 0, so that row keeps its values) at the end of the step
// before.  With p = ks kW + wi, every slot below ks holds a column left of
// the pivot: the loop over ks is unrolled and those slots drop out at
// compile time.  The other slots are updated without a branch: a column
// left of the pivot has a zero in row p (the update changes nothing), the
// pivot column itself becomes zero off the diagonal (it is not read
// again), and slots past the last column hold zeros.
//
// scratch: 192 floats of shared memory (pivot column, double-buffered, and
// the pivots).  D <= 64.  Every thread of the kW warps that take part calls
// this (tid = 0 .. 32 kW - 1); `sync` is their barrier (the whole block by
// default).  On return R holds X; A is not written.
struct BlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
template <int kW, int kC, typename Sync = BlockSync>
__device__ __forceinline__ void solve_walk_system(const float *A, int sb, float *R, int re, int D, int m,
                                                  float *scratch, int tid, Sync sync = Sync()) {
    const int w = tid >> 5, l = tid & 31;
    const bool h0 = l < D, h1 = l + 32 < D;
    const int NC = D + m;
    float *colbuf = scratch, *pivs = scratch + 128;
    float x0[kC], x1[kC];
#pragma unroll
    for (int k = 0; k < kC; ++k) {
        const int c = w + k * kW;
        const float *col = c < D ? A + c * sb : R + (c - D) * re;
        x0[k] = (c < NC && h0) ? col[l] : 0.f;
        x1[k] = (c < NC && h1) ? col[l + 32] : 0.f;
    }
    if (w == 0) {   // pivot column 0: warp 0, slot 0
        if (h0) colbuf[l] = l == 0 ? 0.f : x0[0];
        if (h1) colbuf[l + 32] = x1[0];
        if (l == 0) pivs[0] = x0[0];
    }
    sync();
#pragma unroll
    for (int ks = 0; ks < (64 + kW - 1) / kW; ++ks) {
        for (int wi = 0; wi < kW; ++wi) {
            const int p = ks * kW + wi;
            if (p >= D) break;
            const float *cb = colbuf + (p & 1) * 64;
            float *cn = colbuf + ((p + 1) & 1) * 64;
            const float ipiv = 1.f / pivs[p];
            const float f0 = h0 ? -cb[l] * ipiv : 0.f;
            const float f1 = h1 ? -cb[l + 32] * ipiv : 0.f;
            // pivot row in x1 (rows 32..63)?  Known at compile time unless this ks straddles 32
            const bool hi = ks * kW + kW <= 32 ? false : (ks * kW >= 32 ? true : p >= 32);
            const int src = p & 31;
#pragma unroll
            for (int k = ks; k < kC; ++k) {
                const float pr = __shfl_sync(0xffffffffu, hi ? x1[k] : x0[k], src);
                x0[k] = fmaf(f0, pr, x0[k]);
                x1[k] = fmaf(f1, pr, x1[k]);
            }
            // publish column p + 1 from its owner: warp (p + 1) mod kW, slot ks or ks + 1
            const int pn = p + 1;
            if (pn < D && w == (wi + 1) % kW) {
                const int kn1 = ks + 1 < kC ? ks + 1 : ks;   // static once unrolled: no local arrays
                const bool same = wi + 1 < kW;
                const float y0 = same ? x0[ks] : x0[kn1], y1 = same ? x1[ks] : x1[kn1];
                if (h0) cn[l] = l == pn ? 0.f : y0;
                if (h1) cn[l + 32] = l + 32 == pn ? 0.f : y1;
                if (l == (pn & 31)) pivs[pn] = pn < 32 ? y0 : y1;
            }
            sync();
        }
    }
    // X = (transformed R) / pivot, row by row, back into R
    const float d0 = h0 ? pivs[l] : 1.f, d1 = h1 ? pivs[l + 32] : 1.f;
#pragma unroll
    for (int k = 0; k < kC; ++k) {
        const int c = w + k * kW;
        if (c >= D && c < NC) {
            float *col = R + (c - D) * re;
            if (h0) col[l] = x0[k] / d0;
            if (h1) col[l + 32] = x1[k] / d1;
        }
    }
    sync();
}

}  // namespace lisa
