/*
 * lisa_oracle.c -- plain double-precision CPU oracle of the LiSA layer: its
 * forward and its backward (the gradients of the inputs, of alpha and of the
 * MLP's parameters).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it is written straight from the method's definition.
 *
 * Source: "LiSA: Linear Stochastic Attention for Long-Range Visual Modeling"
 * (reading note of arXiv 2611.04216v2, cc.laoqi.cc), cited below as [note].
 *   [note §2.1]  token set, projections, ReLU feature map (paper Table 8)
 *   [note §2.2]  row-stochastic transition S = Q~ K^T, geometric truncated
 *                walk weights (paper Sec. 3.2, Eq. 4)
 *   [note §2.3]  low-rank evaluation S^k V = Q~ (K^T Q~)^(k-1) K^T V
 *                (paper Eq. 8, Algorithm 1)
 *   [note §2.4]  adaptive per-token, per-head step weights from a 2-layer
 *                MLP + softmax (paper Eq. 10, Supp. Sec. 8); the 3x3 local
 *                branch and the alpha mix (paper Sec. 3.2, Fig. 2)
 *
 * The display equations were lost when the note was extracted, so a few
 * details are readings, stated where they are used:
 *   - Q~_i = Q_i / (Q_i . sum_j K_j + eps), the sum running over every token.
 *   - walk index k = 0..T-1 with k = 0 the identity (T = 1 keeps only S^0 = I).
 *   - MLP input is concat(q_i, k_i) of the feature-mapped (post-ReLU) query
 *     and key; hidden layer has a bias and the exact erf GELU; the output
 *     layer has a bias; softmax over the T logits with the max subtracted.
 *   - local branch: scores q_i . k_j / sqrt(d_h) over the token itself and its
 *     in-grid 8-neighbours (neighbours outside the grid are left out, not
 *     zero-padded), softmax over those, applied to V.
 *   - alpha is used as given, one value per head.
 *
 * Untruncated walk (T = 0 with geometric weights): the note (§2.3, the
 * closing remark on the geometric series) observes that without truncation
 * the series has a closed form; with weights (1-beta) beta^k for every k >= 0
 * it is g = (1-beta) (I - beta S)^(-1) V.
 *
 * Two evaluation modes give the same global branch by different routes:
 *   EXPLICIT: rows of S are formed one at a time and Y_k = S Y_(k-1) is
 *             iterated over n x n products (O(T n^2 d)); S is never stored.
 *   LOWRANK:  s, M = K^T Q~, U_1 = K^T V, U_k = M U_(k-1), Y_k = Q~ U_k.
 * and, for the untruncated walk,
 *   EXPLICIT: the n x n system (I - beta S) X = V solved densely;
 *   LOWRANK:  (I - beta Q~ K^T)^(-1) = I + beta Q~ (I - beta M)^(-1) K^T (the
 *             push-through identity, a derivation of ours, not the note's), so
 *             g = (1-beta) (V + beta Q~ Z) with (I - beta M) Z = U_1, d x d.
 *
 * Feature maps (the fmap argument, "relu_inputs"): none, ReLU, or ELU(x) + 1,
 * the reading taken of the note's ELU variant (§2.1; paper Table 8).
 *
 * The backward (lisa_oracle_backward) is the chain rule written out by hand
 * through the forward's steps in reverse; the derivation sits above
 * backward_slice and mlp_walk_backward.
 *
 * Every array is row-major, double precision, contiguous:
 *   Q, K  [B][heads][n][d_h]      V, O, G, L  [B][heads][n][d_v]
 * with n = H*W and token index i = r*W + c on the H x W grid.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EXPLICIT 0
#define ORACLE_LOWRANK 1

#define ORACLE_W_GEOMETRIC 0
#define ORACLE_W_FIXED 1
#define ORACLE_W_MLP 2
#define ORACLE_MAX_T 256
#define ORACLE_MAX_HIDDEN 1024

/* OpenMP only spreads independent outputs (query rows, matrix entries,
 * tokens) over threads; every sum keeps its serial order. */
static int omp_thread(void)
{
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

static int omp_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* Walk weights, [note §2.2] (paper Eq. 4): a walk continues with          */
/* probability beta; the weight of length k is (1-beta) beta^k, and the     */
/* first T weights are renormalised by their sum 1 - beta^T.                */
/* ---------------------------------------------------------------------- */
int lisa_oracle_geometric_weights(double beta, int T, double *w)
{
    if (T < 1 || !(beta >= 0.0) || !(beta < 1.0)) return 1;
    double norm = 1.0 - pow(beta, (double)T);
    for (int k = 0; k < T; ++k)
        w[k] = (1.0 - beta) * pow(beta, (double)k) / norm;
    return 0;
}

/* Feature map [note §2.1]: the argument `fmap` of every entry point is
 *   0  none: the inputs are the features (already non-negative);
 *   1  ReLU: Q = max(Xq, 0), K = max(Xk, 0) (the paper's default);
 *   2  ELU + 1: phi(x) = x + 1 for x > 0, exp(x) otherwise.  The note (§2.1;
 *      paper Table 8) compares an ELU feature map with ReLU; the non-negative
 *      form ELU(x) + 1 is the reading taken, since the transition S must stay
 *      non-negative and row-stochastic. */
#define ORACLE_FMAP_NONE 0
#define ORACLE_FMAP_RELU 1
#define ORACLE_FMAP_ELU1 2

static double feature_value(double x, int fmap)
{
    if (fmap == ORACLE_FMAP_RELU) return x < 0.0 ? 0.0 : x;
    if (fmap == ORACLE_FMAP_ELU1) return x > 0.0 ? x + 1.0 : exp(x);
    return x;
}

/* d phi / dx at x (the backward's mask or scale). */
static double feature_slope(double x, int fmap)
{
    if (fmap == ORACLE_FMAP_RELU) return x > 0.0 ? 1.0 : 0.0;
    if (fmap == ORACLE_FMAP_ELU1) return x > 0.0 ? 1.0 : exp(x);
    return 1.0;
}

static void feature_map(const double *X, double *out, long count, int fmap)
{
    for (long t = 0; t < count; ++t) out[t] = feature_value(X[t], fmap);
}

/* s = sum over every token j of K_j  [note §2.2]. */
static void key_sum(const double *K, int n, int dh, double *s)
{
    for (int a = 0; a < dh; ++a) s[a] = 0.0;
    for (int j = 0; j < n; ++j)
        for (int a = 0; a < dh; ++a) s[a] += K[(long)j * dh + a];
}

/* Q~_i = Q_i / (Q_i . s + eps)  [note §2.2]. */
static void normalised_queries(const double *Q, const double *s, int n, int dh,
                               double eps, double *Qt)
{
    for (int i = 0; i < n; ++i) {
        const double *q = Q + (long)i * dh;
        double den = eps;
        for (int a = 0; a < dh; ++a) den += q[a] * s[a];
        for (int a = 0; a < dh; ++a) Qt[(long)i * dh + a] = q[a] / den;
    }
}

/* ---------------------------------------------------------------------- */
/* Global branch, EXPLICIT mode: Y_0 = V, Y_k = S Y_(k-1) with             */
/* S_ij = Q~_i . K_j formed on the fly.  Writes Y_0..Y_(T-1) into          */
/* Y[T][n][dv].                                                             */
/* ---------------------------------------------------------------------- */
static void walk_terms_explicit(const double *Qt, const double *K,
                                const double *V, int n, int dh, int dv, int T,
                                double *Y, double *Srows)
{
    memcpy(Y, V, sizeof(double) * (size_t)n * dv);
    for (int k = 1; k < T; ++k) {
        const double *prev = Y + (size_t)(k - 1) * n * dv;
        double *cur = Y + (size_t)k * n * dv;
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i) {
            double *Srow = Srows + (size_t)omp_thread() * n;
            for (int j = 0; j < n; ++j) {
                double sij = 0.0;
                for (int a = 0; a < dh; ++a)
                    sij += Qt[(long)i * dh + a] * K[(long)j * dh + a];
                Srow[j] = sij;
            }
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int j = 0; j < n; ++j) acc += Srow[j] * prev[(long)j * dv + e];
                cur[(long)i * dv + e] = acc;
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Global branch, LOWRANK mode [note §2.3] (paper Eq. 8, Algorithm 1):      */
/* for k >= 1, S^k V = Q~ (K^T Q~)^(k-1) (K^T V).                           */
/*   M   = K^T Q~            (dh x dh)                                      */
/*   U_1 = K^T V             (dh x dv)                                      */
/*   U_k = M U_(k-1)                                                        */
/*   Y_k = Q~ U_k            (n x dv),  Y_0 = V                             */
/* ---------------------------------------------------------------------- */
static void walk_terms_lowrank(const double *Qt, const double *K,
                               const double *V, int n, int dh, int dv, int T,
                               double *Y, double *M, double *U, double *Unext)
{
    memcpy(Y, V, sizeof(double) * (size_t)n * dv);
    if (T < 2) return;
#pragma omp parallel for collapse(2) schedule(static)
    for (int a = 0; a < dh; ++a)
        for (int b = 0; b < dh; ++b) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * Qt[(long)j * dh + b];
            M[a * dh + b] = acc;
        }
#pragma omp parallel for collapse(2) schedule(static)
    for (int a = 0; a < dh; ++a)
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * V[(long)j * dv + e];
            U[a * dv + e] = acc;
        }
    for (int k = 1; k < T; ++k) {
        if (k > 1) {
            for (int a = 0; a < dh; ++a)
                for (int e = 0; e < dv; ++e) {
                    double acc = 0.0;
                    for (int b = 0; b < dh; ++b) acc += M[a * dh + b] * U[b * dv + e];
                    Unext[a * dv + e] = acc;
                }
            memcpy(U, Unext, sizeof(double) * (size_t)dh * dv);
        }
        double *cur = Y + (size_t)k * n * dv;
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i)
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int a = 0; a < dh; ++a) acc += Qt[(long)i * dh + a] * U[a * dv + e];
                cur[(long)i * dv + e] = acc;
            }
    }
}

/* ---------------------------------------------------------------------- */
/* Dense linear solve A X = R (A: n x n, R: n x m, row-major; both are      */
/* overwritten, X is left in R) by Gaussian elimination with partial        */
/* pivoting and back substitution.  Returns 3 for a singular A.             */
/* ---------------------------------------------------------------------- */
static int solve_dense(double *A, double *R, int n, int m)
{
    for (int p = 0; p < n; ++p) {
        int piv = p;
        double best = fabs(A[(long)p * n + p]);
        for (int i = p + 1; i < n; ++i)
            if (fabs(A[(long)i * n + p]) > best) {
                best = fabs(A[(long)i * n + p]);
                piv = i;
            }
        if (!(best > 0.0)) return 3;
        if (piv != p) {
            for (int j = 0; j < n; ++j) {
                double t = A[(long)p * n + j];
                A[(long)p * n + j] = A[(long)piv * n + j];
                A[(long)piv * n + j] = t;
            }
            for (int e = 0; e < m; ++e) {
                double t = R[(long)p * m + e];
                R[(long)p * m + e] = R[(long)piv * m + e];
                R[(long)piv * m + e] = t;
            }
        }
#pragma omp parallel for schedule(static)
        for (int i = p + 1; i < n; ++i) {
            const double f = A[(long)i * n + p] / A[(long)p * n + p];
            A[(long)i * n + p] = 0.0;
            for (int j = p + 1; j < n; ++j) A[(long)i * n + j] -= f * A[(long)p * n + j];
            for (int e = 0; e < m; ++e) R[(long)i * m + e] -= f * R[(long)p * m + e];
        }
    }
    for (int p = n - 1; p >= 0; --p)
        for (int e = 0; e < m; ++e) {
            double acc = R[(long)p * m + e];
            for (int j = p + 1; j < n; ++j) acc -= A[(long)p * n + j] * R[(long)j * m + e];
            R[(long)p * m + e] = acc / A[(long)p * n + p];
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Untruncated geometric walk: g = (1-beta) sum_{k>=0} beta^k S^k V         */
/*                               = (1-beta) (I - beta S)^(-1) V.            */
/* EXPLICIT solves the n x n system; LOWRANK the d x d one of the           */
/* push-through identity, g = (1-beta) (V + beta Q~ Z), (I - beta M) Z = U_1.*/
/* ---------------------------------------------------------------------- */
static int walk_untruncated(const double *Qt, const double *K, const double *V, int n,
                            int dh, int dv, double beta, int mode, double *g)
{
    int err = 0;
    if (mode == ORACLE_EXPLICIT) {
        double *A = malloc(sizeof(double) * (size_t)n * n);
        if (!A) return 2;
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double sij = 0.0;
                for (int a = 0; a < dh; ++a) sij += Qt[(long)i * dh + a] * K[(long)j * dh + a];
                A[(long)i * n + j] = (i == j ? 1.0 : 0.0) - beta * sij;
            }
        memcpy(g, V, sizeof(double) * (size_t)n * dv);
        err = solve_dense(A, g, n, dv);
        for (long t = 0; t < (long)n * dv; ++t) g[t] *= 1.0 - beta;
        free(A);
        return err;
    }
    double *A = malloc(sizeof(double) * (size_t)dh * dh);
    double *Z = malloc(sizeof(double) * (size_t)dh * dv);
    if (!A || !Z) { free(A); free(Z); return 2; }
    for (int a = 0; a < dh; ++a)
        for (int b = 0; b < dh; ++b) {
            double acc = 0.0;   /* M_ab = sum_j K_j[a] Q~_j[b] */
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * Qt[(long)j * dh + b];
            A[a * dh + b] = (a == b ? 1.0 : 0.0) - beta * acc;
        }
    for (int a = 0; a < dh; ++a)
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;   /* (U_1)_ae = sum_j K_j[a] V_j[e] */
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * V[(long)j * dv + e];
            Z[a * dv + e] = acc;
        }
    err = solve_dense(A, Z, dh, dv);
    if (!err) {
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i)
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int a = 0; a < dh; ++a) acc += Qt[(long)i * dh + a] * Z[a * dv + e];
                g[(long)i * dv + e] = (1.0 - beta) * (V[(long)i * dv + e] + beta * acc);
            }
    }
    free(A); free(Z);
    return err;
}

/* ---------------------------------------------------------------------- */
/* Adaptive step weights [note §2.4] (paper Eq. 10, Supp. Sec. 8):          */
/* x = concat(q_i, k_i);  h = GELU(W1 x + b1);  z = W2 h + b2;              */
/* w(i) = softmax(z) over the T walk lengths.  W1 is [hidden][2*dh] and     */
/* W2 is [T][hidden] (output-major, like a torch Linear weight).           */
/* ---------------------------------------------------------------------- */
static double gelu_erf(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

static void mlp_step_weights(const double *q, const double *k, int dh, int T,
                             const double *W1, const double *b1,
                             const double *W2, const double *b2, int hidden,
                             double *h, double *w)
{
    for (int m = 0; m < hidden; ++m) {
        const double *row = W1 + (long)m * 2 * dh;
        double acc = b1[m];
        for (int a = 0; a < dh; ++a) acc += row[a] * q[a];
        for (int a = 0; a < dh; ++a) acc += row[dh + a] * k[a];
        h[m] = gelu_erf(acc);
    }
    double zmax = -INFINITY;
    for (int t = 0; t < T; ++t) {
        double acc = b2[t];
        for (int m = 0; m < hidden; ++m) acc += W2[(long)t * hidden + m] * h[m];
        w[t] = acc;
        if (acc > zmax) zmax = acc;
    }
    double sum = 0.0;
    for (int t = 0; t < T; ++t) {
        w[t] = exp(w[t] - zmax);
        sum += w[t];
    }
    for (int t = 0; t < T; ++t) w[t] /= sum;
}

/* ---------------------------------------------------------------------- */
/* Local 3x3 branch [note §2.4] (paper Sec. 3.2): for token i at (r, c) the  */
/* window is every in-grid (r+dr, c+dc), dr, dc in {-1, 0, 1}: the token     */
/* itself plus at most 8 neighbours.  e_ij = q_i . k_j / sqrt(dh); the       */
/* weights are exp(e_ij - max_j e_ij) normalised over the window.           */
/* ---------------------------------------------------------------------- */
static void local_branch(const double *Qf, const double *Kf, const double *V,
                         int H, int W, int dh, int dv, double *L)
{
    const double scale = 1.0 / sqrt((double)dh);
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < H; ++r)
        for (int c = 0; c < W; ++c) {
            int i = r * W + c;
            int nb[9], cnt = 0;
            double e[9];
            for (int dr = -1; dr <= 1; ++dr)
                for (int dc = -1; dc <= 1; ++dc) {
                    int rr = r + dr, cc = c + dc;
                    if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue;
                    nb[cnt++] = rr * W + cc;
                }
            double emax = -INFINITY;
            for (int t = 0; t < cnt; ++t) {
                double acc = 0.0;
                for (int a = 0; a < dh; ++a)
                    acc += Qf[(long)i * dh + a] * Kf[(long)nb[t] * dh + a];
                e[t] = acc * scale;
                if (e[t] > emax) emax = e[t];
            }
            double den = 0.0;
            for (int t = 0; t < cnt; ++t) {
                e[t] = exp(e[t] - emax);
                den += e[t];
            }
            for (int x = 0; x < dv; ++x) {
                double acc = 0.0;
                for (int t = 0; t < cnt; ++t) acc += e[t] * V[(long)nb[t] * dv + x];
                L[(long)i * dv + x] = acc / den;
            }
        }
}

/* ---------------------------------------------------------------------- */
/* One (batch, head) slice: feature map, global walk, weights, local branch, */
/* alpha mix  o = alpha * g + (1 - alpha) * l  [note §2.4] (paper Fig. 2).   */
/* ---------------------------------------------------------------------- */
typedef struct {
    int H, W, dh, dv, T, wmode, hidden, mode, relu;   /* T = 0: untruncated walk; relu: the fmap */
    double eps, beta;
    const double *w, *W1, *b1, *W2, *b2;
} slice_args;

static int forward_slice(const slice_args *A, const double *Xq, const double *Xk,
                         const double *V, double alpha, double *O, double *G,
                         double *L)
{
    const int n = A->H * A->W, dh = A->dh, dv = A->dv, T = A->T;
    double *Qf = malloc(sizeof(double) * (size_t)n * dh);
    double *Kf = malloc(sizeof(double) * (size_t)n * dh);
    double *Qt = malloc(sizeof(double) * (size_t)n * dh);
    double *Y = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * n * dv);
    double *g = malloc(sizeof(double) * (size_t)n * dv);
    double *l = malloc(sizeof(double) * (size_t)n * dv);
    double *Srows = malloc(sizeof(double) * (size_t)n * omp_threads());
    double *M = malloc(sizeof(double) * (size_t)dh * dh);
    double *U = malloc(sizeof(double) * (size_t)dh * dv);
    double *Un = malloc(sizeof(double) * (size_t)dh * dv);
    double s[256];
    int err = 0;
    if (!Qf || !Kf || !Qt || !Y || !g || !l || !Srows || !M || !U || !Un) {
        err = 2;
        goto done;
    }
    feature_map(Xq, Qf, (long)n * dh, A->relu);
    feature_map(Xk, Kf, (long)n * dh, A->relu);
    key_sum(Kf, n, dh, s);
    normalised_queries(Qf, s, n, dh, A->eps, Qt);
    if (T == 0) {
        err = walk_untruncated(Qt, Kf, V, n, dh, dv, A->beta, A->mode, g);
        if (err) goto done;
    } else if (A->mode == ORACLE_EXPLICIT)
        walk_terms_explicit(Qt, Kf, V, n, dh, dv, T, Y, Srows);
    else
        walk_terms_lowrank(Qt, Kf, V, n, dh, dv, T, Y, M, U, Un);

    /* g_i = sum_k w_k(i) Y_k,i with the token's own weights in MLP mode */
    if (T > 0) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < n; ++i) {
        double wk[ORACLE_MAX_T], h[ORACLE_MAX_HIDDEN];
        if (A->wmode == ORACLE_W_MLP)
            mlp_step_weights(Qf + (long)i * dh, Kf + (long)i * dh, dh, T, A->W1,
                             A->b1, A->W2, A->b2, A->hidden, h, wk);
        else
            for (int k = 0; k < T; ++k) wk[k] = A->w[k];
        for (int x = 0; x < dv; ++x) {
            double acc = 0.0;
            for (int k = 0; k < T; ++k) acc += wk[k] * Y[(size_t)k * n * dv + (long)i * dv + x];
            g[(long)i * dv + x] = acc;
        }
    }
    }
    local_branch(Qf, Kf, V, A->H, A->W, dh, dv, l);
    for (long t = 0; t < (long)n * dv; ++t) {
        if (O) O[t] = alpha * g[t] + (1.0 - alpha) * l[t];
        if (G) G[t] = g[t];
        if (L) L[t] = l[t];
    }
done:
    free(Qf); free(Kf); free(Qt); free(Y); free(g); free(l); free(Srows);
    free(M); free(U); free(Un);
    return err;
}

/*
 * Full layer over B x heads independent slices.
 *   wmode   0 geometric (beta), 1 fixed (w[T]), 2 MLP (W1,b1,W2,b2,hidden)
 *   T       walk truncation depth >= 1; 0 with geometric weights: untruncated
 *   alpha   [heads]
 *   mode    0 EXPLICIT, 1 LOWRANK
 *   relu_inputs  the feature map: 0 none, 1 ReLU, 2 ELU + 1
 *   O, G, L may each be NULL; G and L receive the global and local branches.
 *   nthreads <= 0 uses the OpenMP default.
 * Returns 0 on success, 1 on a bad argument, 2 on allocation failure, 3 when
 * an untruncated walk meets a singular system.
 */
int lisa_oracle_forward(const double *Xq, const double *Xk, const double *V,
                        double *O, double *G, double *L, int B, int heads,
                        int H, int W, int dh, int dv, int T, int wmode,
                        double beta, const double *w, const double *W1,
                        const double *b1, const double *W2, const double *b2,
                        int hidden, const double *alpha, double eps,
                        int relu_inputs, int mode, int nthreads)
{
    if (B < 0 || heads < 0 || H < 1 || W < 1 || dh < 1 || dh > 256 || dv < 1 || T < 0 ||
        T > ORACLE_MAX_T)
        return 1;
    if (eps < 0.0 || !alpha || relu_inputs < 0 || relu_inputs > 2) return 1;
    if (T == 0 && (wmode != ORACLE_W_GEOMETRIC || !(beta >= 0.0) || !(beta < 1.0))) return 1;
    double *wts = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    if (!wts) return 2;
    if (T == 0) {
        wts[0] = 1.0 - beta;   /* w_0 of the untruncated walk; the hops go through the solve */
    } else if (wmode == ORACLE_W_GEOMETRIC) {
        if (lisa_oracle_geometric_weights(beta, T, wts)) { free(wts); return 1; }
    } else if (wmode == ORACLE_W_FIXED) {
        if (!w) { free(wts); return 1; }
        memcpy(wts, w, sizeof(double) * (size_t)T);
    } else if (wmode == ORACLE_W_MLP) {
        if (!W1 || !b1 || !W2 || !b2 || hidden < 1 || hidden > ORACLE_MAX_HIDDEN) {
            free(wts);
            return 1;
        }
    } else {
        free(wts);
        return 1;
    }
    slice_args A = {H, W, dh, dv, T, wmode, hidden, mode, relu_inputs, eps, beta,
                    wts, W1, b1, W2, b2};
    const long n = (long)H * W;
    const long slices = (long)B * heads;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    for (long sl = 0; sl < slices; ++sl) {
        long hq = sl * n * dh, hv = sl * n * dv;
        const int e = forward_slice(&A, Xq + hq, Xk + hq, V + hv, alpha[sl % heads],
                                    O ? O + hv : NULL, G ? G + hv : NULL, L ? L + hv : NULL);
        if (e && !err) err = e;
    }
    free(wts);
    return err;
}

/* ---------------------------------------------------------------------- */
/* Backward pass of one slice with fixed walk weights (geometric resolved   */
/* to fixed), by the chain rule through the forward above, in the order of  */
/* the forward's steps taken backwards.  Given dO = dL/dO:                  */
/*   o = alpha g + (1-alpha) l:  dalpha = sum_i dO_i . (g_i - l_i),         */
/*                               dg = alpha dO,  dl = (1-alpha) dO          */
/*   g_i = w_0 V_i + Q~_i Ubar, Ubar = sum_{k>=1} w_k U_k:                  */
/*        dV += w_0 dg,  dQ~ = dg Ubar^T,  dUbar = Q~^T dg                  */
/*   U_k = M U_(k-1):  G_(T-1) = w_(T-1) dUbar, G_k = w_k dUbar + M^T G_(k+1)*/
/*        (G_k = dL/dU_k),  dM = sum_{k>=2} G_k U_(k-1)^T,  dU_1 = G_1      */
/*   U_1 = K^T V:  dK_j += dU_1 V_j,  dV_j += dU_1^T K_j                    */
/*   M = K^T Q~:   dK_j += dM Q~_j,   dQ~_j += dM^T K_j                     */
/*   Q~_i = Q_i / r_i, r_i = Q_i . s + eps:  c_i = (dQ~_i . Q~_i) / r_i,    */
/*        dQ_i += dQ~_i / r_i - c_i s,  ds = -sum_i c_i Q_i                 */
/*   s = sum_j K_j:  dK_j += ds                                             */
/*   local, e_ij = q_i . k_j / sqrt(dh), a = softmax_j, l_i = sum a_ij V_j: */
/*        dV_j += a_ij dl_i,  de_ij = a_ij (dl_i . V_j - dl_i . l_i),       */
/*        dQ_i += sum_j de_ij K_j / sqrt(dh), dK_j += de_ij Q_i / sqrt(dh)  */
/*   feature map: dXq = dQ [Xq > 0], dXk = dK [Xk > 0] (relu set).          */
/* Untruncated walk (T = 0): Ubar = beta (1-beta) Z, (I - beta M) Z = U_1,  */
/*   so with A = I - beta M and dZ = beta (1-beta) dUbar:                   */
/*   dU_1 = A^-T dZ,  dM = beta (A^-T dZ) Z^T, and w_0 = 1 - beta.           */
/* ---------------------------------------------------------------------- */
/* GELU (exact erf form) and its derivative 0.5 (1 + erf(a/sqrt 2)) + a phi(a). */
static double gelu_erf_grad(double a)
{
    const double pi = 3.14159265358979323846;
    return 0.5 * (1.0 + erf(a / sqrt(2.0))) + a * exp(-0.5 * a * a) / sqrt(2.0 * pi);
}

/* ---------------------------------------------------------------------- */
/* Global branch of the backward pass with the adaptive (per-token) walk    */
/* weights [note §2.4] (paper Eq. 10, Supp. Sec. 8).  Forward, per token i: */
/*   x_i = [q_i; k_i], a_i = W1 x_i + b1, h_i = GELU(a_i), z_i = W2 h_i + b2,*/
/*   w_i = softmax(z_i),  g_i = w_i0 V_i + sum_{k>=1} w_ik Y_k,i,            */
/*   Y_k = Q~ U_k.  Backward, with dg = alpha dO:                           */
/*   dw_ik = dg_i . Y_k,i (Y_0 = V);  dz_i = w_i (dw_i - w_i . dw_i);       */
/*   dW2 += dz_i h_i^T, db2 += dz_i;  da_i = (W2^T dz_i) GELU'(a_i);        */
/*   dW1 += da_i x_i^T, db1 += da_i;  [dq_i; dk_i] += W1^T da_i  (the MLP's */
/*   share of the feature gradients);                                       */
/*   dV_i = w_i0 dg_i;  dQ~_i = sum_{k>=1} w_ik dg_i U_k^T;                 */
/*   dU_k = sum_i Q~_i (w_ik dg_i)^T;  G_(T-1) = dU_(T-1),                  */
/*   G_k = dU_k + M^T G_(k+1), dM = sum_{k>=2} G_k U_(k-1)^T, dU_1 = G_1.   */
/* Writes g, dV, dQ~, dM, dU_1, the MLP's feature gradients dqm, dkm, and   */
/* adds the parameter gradients into dW1, db1, dW2, db2.                    */
/* ---------------------------------------------------------------------- */
static int mlp_walk_backward(const slice_args *A, const double *Q, const double *K, const double *Qt,
                             const double *V, const double *dO, double alpha, const double *M,
                             const double *Uk, double *g, double *dV, double *dQt, double *dM,
                             double *dU1, double *dqm, double *dkm, double *dW1, double *db1,
                             double *dW2, double *db2)
{
    const int n = A->H * A->W, dh = A->dh, dv = A->dv, T = A->T, hid = A->hidden;
    const size_t dd = (size_t)dh * dv;
    double *wt = malloc(sizeof(double) * (size_t)n * T), *pre = malloc(sizeof(double) * (size_t)n * hid);
    double *hh = malloc(sizeof(double) * (size_t)n * hid), *dUk = calloc((size_t)(T > 1 ? T - 1 : 1) * dd, sizeof(double));
    double *G = malloc(sizeof(double) * (size_t)(T > 1 ? T - 1 : 1) * dd);
    double *Y = malloc(sizeof(double) * (size_t)T * dv), *dw = malloc(sizeof(double) * (size_t)T);
    double *dz = malloc(sizeof(double) * (size_t)T), *da = malloc(sizeof(double) * (size_t)hid);
    int err = 0;
    if (!wt || !pre || !hh || !dUk || !G || !Y || !dw || !dz || !da) {
        err = 2;
        goto out;
    }
    for (int i = 0; i < n; ++i) {
        const double *q = Q + (long)i * dh, *k = K + (long)i * dh;
        /* forward through the MLP, keeping the pre-activations */
        for (int m = 0; m < hid; ++m) {
            const double *row = A->W1 + (long)m * 2 * dh;
            double acc = A->b1[m];
            for (int c = 0; c < dh; ++c) acc += row[c] * q[c] + row[dh + c] * k[c];
            pre[(long)i * hid + m] = acc;
            hh[(long)i * hid + m] = gelu_erf(acc);
        }
        double zmax = -INFINITY, zs = 0.0;
        double *w = wt + (long)i * T;
        for (int t = 0; t < T; ++t) {
            double acc = A->b2[t];
            for (int m = 0; m < hid; ++m) acc += A->W2[(long)t * hid + m] * hh[(long)i * hid + m];
            w[t] = acc;
            if (acc > zmax) zmax = acc;
        }
        for (int t = 0; t < T; ++t) {
            w[t] = exp(w[t] - zmax);
            zs += w[t];
        }
        for (int t = 0; t < T; ++t) w[t] /= zs;
        /* walk terms Y_k,i and the token's global value */
        for (int e = 0; e < dv; ++e) Y[e] = V[(long)i * dv + e];
        for (int kk = 1; kk < T; ++kk)
            for (int e = 0; e < dv; ++e) {
                double acc = 0.0;
                for (int a = 0; a < dh; ++a) acc += Qt[(long)i * dh + a] * Uk[(size_t)(kk - 1) * dd + a * dv + e];
                Y[(size_t)kk * dv + e] = acc;
            }
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += w[t] * Y[(size_t)t * dv + e];
            g[(long)i * dv + e] = acc;
        }
        /* weights: dw, dz through the softmax */
        double wdw = 0.0;
        for (int t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int e = 0; e < dv; ++e) acc += alpha * dO[(long)i * dv + e] * Y[(size_t)t * dv + e];
            dw[t] = acc;
            wdw += w[t] * acc;
        }
        for (int t = 0; t < T; ++t) dz[t] = w[t] * (dw[t] - wdw);
        /* MLP parameters and inputs */
        for (int t = 0; t < T; ++t) {
            db2[t] += dz[t];
            for (int m = 0; m < hid; ++m) dW2[(long)t * hid + m] += dz[t] * hh[(long)i * hid + m];
        }
        for (int m = 0; m < hid; ++m) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += A->W2[(long)t * hid + m] * dz[t];
            da[m] = acc * gelu_erf_grad(pre[(long)i * hid + m]);
            db1[m] += da[m];
            for (int c = 0; c < dh; ++c) {
                dW1[(long)m * 2 * dh + c] += da[m] * q[c];
                dW1[(long)m * 2 * dh + dh + c] += da[m] * k[c];
            }
        }
        for (int c = 0; c < dh; ++c) {
            double aq = 0.0, ak = 0.0;
            for (int m = 0; m < hid; ++m) {
                aq += A->W1[(long)m * 2 * dh + c] * da[m];
                ak += A->W1[(long)m * 2 * dh + dh + c] * da[m];
            }
            dqm[(long)i * dh + c] = aq;
            dkm[(long)i * dh + c] = ak;
        }
        /* the walk terms */
        for (int e = 0; e < dv; ++e) dV[(long)i * dv + e] = w[0] * alpha * dO[(long)i * dv + e];
        for (int a = 0; a < dh; ++a) {
            double acc = 0.0;
            for (int kk = 1; kk < T; ++kk)
                for (int e = 0; e < dv; ++e)
                    acc += w[kk] * alpha * dO[(long)i * dv + e] * Uk[(size_t)(kk - 1) * dd + a * dv + e];
            dQt[(long)i * dh + a] = acc;
        }
        for (int kk = 1; kk < T; ++kk)
            for (int a = 0; a < dh; ++a)
                for (int e = 0; e < dv; ++e)
                    dUk[(size_t)(kk - 1) * dd + a * dv + e] += Qt[(long)i * dh + a] * w[kk] * alpha * dO[(long)i * dv + e];
    }
    memset(dM, 0, sizeof(double) * dh * dh);
    memset(dU1, 0, sizeof(double) * dd);
    if (T > 1) {
        for (int kk = T - 1; kk >= 1; --kk) {
            double *Gk = G + (size_t)(kk - 1) * dd;
            memcpy(Gk, dUk + (size_t)(kk - 1) * dd, sizeof(double) * dd);
            if (kk < T - 1) {
                const double *Gn = G + (size_t)kk * dd;
                for (int a = 0; a < dh; ++a)
                    for (int e = 0; e < dv; ++e) {
                        double acc = 0.0;
                        for (int b = 0; b < dh; ++b) acc += M[b * dh + a] * Gn[b * dv + e];
                        Gk[a * dv + e] += acc;
                    }
            }
        }
        for (int kk = 2; kk < T; ++kk) {
            const double *Gk = G + (size_t)(kk - 1) * dd, *Up = Uk + (size_t)(kk - 2) * dd;
            for (int a = 0; a < dh; ++a)
                for (int b = 0; b < dh; ++b) {
                    double acc = 0.0;
                    for (int e = 0; e < dv; ++e) acc += Gk[a * dv + e] * Up[b * dv + e];
                    dM[a * dh + b] += acc;
                }
        }
        memcpy(dU1, G, sizeof(double) * dd);
    }
out:
    free(wt); free(pre); free(hh); free(dUk); free(G); free(Y); free(dw); free(dz); free(da);
    return err;
}

static int backward_slice(const slice_args *A, const double *Xq, const double *Xk,
                          const double *V, const double *dO, double alpha,
                          double *dXq, double *dXk, double *dV, double *dalpha,
                          double *dW1, double *db1, double *dW2, double *db2)
{
    const int H = A->H, W = A->W, n = H * W, dh = A->dh, dv = A->dv;
    const int T = A->T, nh = T == 0 ? 1 : (T > 1 ? T - 1 : 1);   /* stored U_k */
    const size_t nd = (size_t)n * dh, nv = (size_t)n * dv;
    double *Q = malloc(sizeof(double) * nd), *K = malloc(sizeof(double) * nd);
    double *Qt = malloc(sizeof(double) * nd), *r = malloc(sizeof(double) * n);
    double *M = malloc(sizeof(double) * dh * dh), *Uk = malloc(sizeof(double) * nh * dh * dv);
    double *Ub = malloc(sizeof(double) * dh * dv), *dUb = malloc(sizeof(double) * dh * dv);
    double *G = malloc(sizeof(double) * nh * dh * dv), *dM = malloc(sizeof(double) * dh * dh);
    double *dU1 = malloc(sizeof(double) * dh * dv), *Amat = malloc(sizeof(double) * dh * dh);
    double *g = malloc(sizeof(double) * nv), *l = malloc(sizeof(double) * nv);
    double *dQt = malloc(sizeof(double) * nd), *dQ = malloc(sizeof(double) * nd);
    double *dK = malloc(sizeof(double) * nd);
    double *dqm = NULL, *dkm = NULL;   /* the MLP's share of dQ, dK (adaptive weights) */
    const int mlp = A->wmode == ORACLE_W_MLP;
    double s[256], ds[256];
    const double scale = 1.0 / sqrt((double)dh);
    int err = 0;
    if (!Q || !K || !Qt || !r || !M || !Uk || !Ub || !dUb || !G || !dM || !dU1 || !Amat || !g || !l ||
        !dQt || !dQ || !dK) {
        err = 2;
        goto done;
    }
    /* ---- forward quantities */
    feature_map(Xq, Q, (long)nd, A->relu);
    feature_map(Xk, K, (long)nd, A->relu);
    key_sum(K, n, dh, s);
    for (int i = 0; i < n; ++i) {
        double den = A->eps;
        for (int a = 0; a < dh; ++a) den += Q[(long)i * dh + a] * s[a];
        r[i] = den;
        for (int a = 0; a < dh; ++a) Qt[(long)i * dh + a] = Q[(long)i * dh + a] / den;
    }
    for (int a = 0; a < dh; ++a)
        for (int b = 0; b < dh; ++b) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * Qt[(long)j * dh + b];
            M[a * dh + b] = acc;
        }
    for (int a = 0; a < dh; ++a)   /* U_1 into Uk[0] */
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += K[(long)j * dh + a] * V[(long)j * dv + e];
            Uk[a * dv + e] = acc;
        }
    const double w0 = T == 0 ? 1.0 - A->beta : (mlp ? 0.0 : A->w[0]);
    memset(Ub, 0, sizeof(double) * dh * dv);
    if (T == 0) {
        /* Z = (I - beta M)^-1 U_1 into Uk[0]; Ubar = beta (1-beta) Z */
        for (int a = 0; a < dh; ++a)
            for (int b = 0; b < dh; ++b) Amat[a * dh + b] = (a == b ? 1.0 : 0.0) - A->beta * M[a * dh + b];
        if ((err = solve_dense(Amat, Uk, dh, dv))) goto done;
        for (int t = 0; t < dh * dv; ++t) Ub[t] = A->beta * (1.0 - A->beta) * Uk[t];
    } else {
        for (int k = 1; k < T; ++k) {
            double *cur = Uk + (size_t)(k - 1) * dh * dv;
            if (k > 1) {
                const double *prev = Uk + (size_t)(k - 2) * dh * dv;
                for (int a = 0; a < dh; ++a)
                    for (int e = 0; e < dv; ++e) {
                        double acc = 0.0;
                        for (int b = 0; b < dh; ++b) acc += M[a * dh + b] * prev[b * dv + e];
                        cur[a * dv + e] = acc;
                    }
            }
            if (!mlp)
                for (int t = 0; t < dh * dv; ++t) Ub[t] += A->w[k] * cur[t];
        }
    }
    if (mlp) {
        /* per-token weights: g, dV, dQ~, dM, dU_1 and the MLP's gradients at once */
        dqm = malloc(sizeof(double) * nd);
        dkm = malloc(sizeof(double) * nd);
        if (!dqm || !dkm) { err = 2; goto done; }
        if ((err = mlp_walk_backward(A, Q, K, Qt, V, dO, alpha, M, Uk, g, dV, dQt, dM, dU1, dqm, dkm,
                                     dW1, db1, dW2, db2)))
            goto done;
    } else {
        for (int i = 0; i < n; ++i)
            for (int e = 0; e < dv; ++e) {
                double acc = w0 * V[(long)i * dv + e];
                for (int a = 0; a < dh; ++a) acc += Qt[(long)i * dh + a] * Ub[a * dv + e];
                g[(long)i * dv + e] = acc;
            }
    }
    local_branch(Q, K, V, H, W, dh, dv, l);

    /* ---- mix */
    double da = 0.0;
    for (size_t t = 0; t < nv; ++t) da += dO[t] * (g[t] - l[t]);
    *dalpha += da;
    /* dg = alpha dO, dl = (1-alpha) dO are formed where they are used */

    /* ---- global branch (fixed weights; the adaptive ones were done above) */
    if (mlp) goto stats_tail;
    for (size_t t = 0; t < nv; ++t) dV[t] = w0 * alpha * dO[t];
    for (int i = 0; i < n; ++i)   /* dQ~ = dg Ubar^T */
        for (int a = 0; a < dh; ++a) {
            double acc = 0.0;
            for (int e = 0; e < dv; ++e) acc += alpha * dO[(long)i * dv + e] * Ub[a * dv + e];
            dQt[(long)i * dh + a] = acc;
        }
    for (int a = 0; a < dh; ++a)   /* dUbar = Q~^T dg */
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i) acc += Qt[(long)i * dh + a] * alpha * dO[(long)i * dv + e];
            dUb[a * dv + e] = acc;
        }
    memset(dM, 0, sizeof(double) * dh * dh);
    memset(dU1, 0, sizeof(double) * dh * dv);
    if (T == 0) {
        /* Y = A^-T dZ with dZ = beta (1-beta) dUbar: solve A^T Y = dZ */
        for (int a = 0; a < dh; ++a)
            for (int b = 0; b < dh; ++b) Amat[a * dh + b] = (a == b ? 1.0 : 0.0) - A->beta * M[b * dh + a];
        for (int t = 0; t < dh * dv; ++t) dU1[t] = A->beta * (1.0 - A->beta) * dUb[t];
        if ((err = solve_dense(Amat, dU1, dh, dv))) goto done;
        for (int a = 0; a < dh; ++a)   /* dM = beta Y Z^T */
            for (int b = 0; b < dh; ++b) {
                double acc = 0.0;
                for (int e = 0; e < dv; ++e) acc += dU1[a * dv + e] * Uk[b * dv + e];
                dM[a * dh + b] = A->beta * acc;
            }
    } else if (T > 1) {
        /* G_k for k = T-1 down to 1, stored at G[k-1] */
        for (int k = T - 1; k >= 1; --k) {
            double *Gk = G + (size_t)(k - 1) * dh * dv;
            for (int t = 0; t < dh * dv; ++t) Gk[t] = A->w[k] * dUb[t];
            if (k < T - 1) {
                const double *Gn = G + (size_t)k * dh * dv;
                for (int a = 0; a < dh; ++a)
                    for (int e = 0; e < dv; ++e) {
                        double acc = 0.0;
                        for (int b = 0; b < dh; ++b) acc += M[b * dh + a] * Gn[b * dv + e];
                        Gk[a * dv + e] += acc;
                    }
            }
        }
        for (int k = 2; k < T; ++k) {   /* dM += G_k U_(k-1)^T */
            const double *Gk = G + (size_t)(k - 1) * dh * dv, *Up = Uk + (size_t)(k - 2) * dh * dv;
            for (int a = 0; a < dh; ++a)
                for (int b = 0; b < dh; ++b) {
                    double acc = 0.0;
                    for (int e = 0; e < dv; ++e) acc += Gk[a * dv + e] * Up[b * dv + e];
                    dM[a * dh + b] += acc;
                }
        }
        memcpy(dU1, G, sizeof(double) * dh * dv);
    }
stats_tail:
    for (int j = 0; j < n; ++j) {
        for (int a = 0; a < dh; ++a) {
            double acc = 0.0;   /* dU_1 V_j + dM Q~_j */
            for (int e = 0; e < dv; ++e) acc += dU1[a * dv + e] * V[(long)j * dv + e];
            for (int b = 0; b < dh; ++b) acc += dM[a * dh + b] * Qt[(long)j * dh + b];
            dK[(long)j * dh + a] = acc;
        }
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;   /* dU_1^T K_j */
            for (int a = 0; a < dh; ++a) acc += dU1[a * dv + e] * K[(long)j * dh + a];
            dV[(long)j * dv + e] += acc;
        }
        for (int b = 0; b < dh; ++b) {
            double acc = 0.0;   /* dM^T K_j */
            for (int a = 0; a < dh; ++a) acc += dM[a * dh + b] * K[(long)j * dh + a];
            dQt[(long)j * dh + b] += acc;
        }
    }
    for (int a = 0; a < dh; ++a) ds[a] = 0.0;
    for (int i = 0; i < n; ++i) {
        double c = 0.0;
        for (int a = 0; a < dh; ++a) c += dQt[(long)i * dh + a] * Qt[(long)i * dh + a];
        c /= r[i];
        for (int a = 0; a < dh; ++a) {
            dQ[(long)i * dh + a] = dQt[(long)i * dh + a] / r[i] - c * s[a];
            ds[a] -= c * Q[(long)i * dh + a];
        }
    }
    for (int j = 0; j < n; ++j)
        for (int a = 0; a < dh; ++a) dK[(long)j * dh + a] += ds[a];
    if (mlp)
        for (size_t t = 0; t < nd; ++t) {
            dQ[t] += dqm[t];
            dK[t] += dkm[t];
        }

    /* ---- local branch */
    for (int rr = 0; rr < H; ++rr)
        for (int cc = 0; cc < W; ++cc) {
            const int i = rr * W + cc;
            int nb[9], cnt = 0;
            double e[9];
            for (int dr = -1; dr <= 1; ++dr)
                for (int dc = -1; dc <= 1; ++dc) {
                    const int r2 = rr + dr, c2 = cc + dc;
                    if (r2 < 0 || r2 >= H || c2 < 0 || c2 >= W) continue;
                    nb[cnt++] = r2 * W + c2;
                }
            double emax = -INFINITY, den = 0.0;
            for (int t = 0; t < cnt; ++t) {
                double acc = 0.0;
                for (int a = 0; a < dh; ++a) acc += Q[(long)i * dh + a] * K[(long)nb[t] * dh + a];
                e[t] = acc * scale;
                if (e[t] > emax) emax = e[t];
            }
            for (int t = 0; t < cnt; ++t) {
                e[t] = exp(e[t] - emax);
                den += e[t];
            }
            double dll = 0.0;   /* dl_i . l_i */
            for (int x = 0; x < dv; ++x) dll += (1.0 - alpha) * dO[(long)i * dv + x] * l[(long)i * dv + x];
            for (int t = 0; t < cnt; ++t) {
                const double a_ij = e[t] / den;
                const int j = nb[t];
                double dlv = 0.0;   /* dl_i . V_j */
                for (int x = 0; x < dv; ++x) {
                    const double dl = (1.0 - alpha) * dO[(long)i * dv + x];
                    dlv += dl * V[(long)j * dv + x];
                    dV[(long)j * dv + x] += a_ij * dl;
                }
                const double de = a_ij * (dlv - dll) * scale;
                for (int a = 0; a < dh; ++a) {
                    dQ[(long)i * dh + a] += de * K[(long)j * dh + a];
                    dK[(long)j * dh + a] += de * Q[(long)i * dh + a];
                }
            }
        }

    /* ---- feature map */
    for (size_t t = 0; t < nd; ++t) {
        dXq[t] = feature_slope(Xq[t], A->relu) * dQ[t];
        dXk[t] = feature_slope(Xk[t], A->relu) * dK[t];
    }
done:
    free(Q); free(K); free(Qt); free(r); free(M); free(Uk); free(Ub); free(dUb); free(G);
    free(dM); free(dU1); free(Amat); free(g); free(l); free(dQt); free(dQ); free(dK);
    free(dqm); free(dkm);
    return err;
}

/*
 * Backward pass of the layer over B x heads slices: dL/dXq, dL/dXk, dL/dV
 * ([B][heads][n][d], overwritten) and dL/dalpha ([heads], overwritten: the
 * sum over the batch) for the upstream gradient dO.  Walk weights as for
 * lisa_oracle_forward: geometric (T >= 1, or T = 0 untruncated), fixed, or
 * adaptive (MLP; then dW1 [hidden][2 dh], db1 [hidden], dW2 [T][hidden], db2
 * [T] are overwritten with the parameter gradients summed over every slice;
 * they may be NULL otherwise).
 */
int lisa_oracle_backward(const double *Xq, const double *Xk, const double *V,
                         const double *dO, double *dXq, double *dXk, double *dV,
                         double *dalpha, int B, int heads, int H, int W, int dh, int dv,
                         int T, int wmode, double beta, const double *w,
                         const double *W1, const double *b1, const double *W2,
                         const double *b2, int hidden, double *dW1, double *db1,
                         double *dW2, double *db2, const double *alpha, double eps,
                         int relu_inputs)
{
    if (B < 0 || heads < 1 || H < 1 || W < 1 || dh < 1 || dh > 256 || dv < 1 || T < 0 ||
        T > ORACLE_MAX_T || eps < 0.0 || !alpha || relu_inputs < 0 || relu_inputs > 2)
        return 1;
    if (T == 0 && wmode != ORACLE_W_GEOMETRIC) return 1;
    if (wmode == ORACLE_W_MLP && (T < 1 || !W1 || !b1 || !W2 || !b2 || hidden < 1 ||
                                  hidden > ORACLE_MAX_HIDDEN || !dW1 || !db1 || !dW2 || !db2))
        return 1;
    double *wts = calloc((size_t)(T > 0 ? T : 1), sizeof(double));
    if (!wts) return 2;
    if (wmode == ORACLE_W_MLP) {
        memset(dW1, 0, sizeof(double) * (size_t)hidden * 2 * dh);
        memset(db1, 0, sizeof(double) * (size_t)hidden);
        memset(dW2, 0, sizeof(double) * (size_t)T * hidden);
        memset(db2, 0, sizeof(double) * (size_t)T);
    } else if (T == 0) {
        if (!(beta >= 0.0 && beta < 1.0)) { free(wts); return 1; }
        wts[0] = 1.0 - beta;
    } else if (wmode == ORACLE_W_GEOMETRIC) {
        if (lisa_oracle_geometric_weights(beta, T, wts)) { free(wts); return 1; }
    } else {
        if (!w) { free(wts); return 1; }
        memcpy(wts, w, sizeof(double) * (size_t)T);
    }
    slice_args A = {H, W, dh, dv, T, wmode, hidden, ORACLE_LOWRANK, relu_inputs, eps, beta,
                    wts, W1, b1, W2, b2};
    const long n = (long)H * W;
    for (int h = 0; h < heads; ++h) dalpha[h] = 0.0;
    int err = 0;
    for (long sl = 0; sl < (long)B * heads; ++sl) {
        const long hq = sl * n * dh, hv = sl * n * dv;
        const int e = backward_slice(&A, Xq + hq, Xk + hq, V + hv, dO + hv, alpha[sl % heads],
                                     dXq + hq, dXk + hq, dV + hv, dalpha + sl % heads, dW1, db1,
                                     dW2, db2);
        if (e && !err) err = e;
    }
    free(wts);
    return err;
}

/*
 * Dense transition matrix of one slice, S_ij = Q~_i . K_j  [note §2.2], for
 * small n only (n x n doubles).  Used by the tests that check that S is
 * non-negative, row-stochastic up to eps and of rank at most dh.
 */
int lisa_oracle_transition(const double *Xq, const double *Xk, int n, int dh,
                           double eps, int relu_inputs, double *S)
{
    if (n < 1 || dh < 1 || dh > 256 || eps < 0.0) return 1;
    double *Qf = malloc(sizeof(double) * (size_t)n * dh);
    double *Kf = malloc(sizeof(double) * (size_t)n * dh);
    double *Qt = malloc(sizeof(double) * (size_t)n * dh);
    double s[256];
    if (!Qf || !Kf || !Qt) { free(Qf); free(Kf); free(Qt); return 2; }
    feature_map(Xq, Qf, (long)n * dh, relu_inputs);
    feature_map(Xk, Kf, (long)n * dh, relu_inputs);
    key_sum(Kf, n, dh, s);
    normalised_queries(Qf, s, n, dh, eps, Qt);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int a = 0; a < dh; ++a) acc += Qt[(long)i * dh + a] * Kf[(long)j * dh + a];
            S[(long)i * n + j] = acc;
        }
    free(Qf); free(Kf); free(Qt);
    return 0;
}

/*
 * Adaptive step weights of every token of one slice [note §2.4]:
 * out[n][T].  Xq, Xk are [n][dh]; the feature map is applied when
 * relu_inputs is set.
 */
int lisa_oracle_step_weights(const double *Xq, const double *Xk, int n, int dh,
                             int T, const double *W1, const double *b1,
                             const double *W2, const double *b2, int hidden,
                             int relu_inputs, double *out)
{
    if (n < 1 || dh < 1 || T < 1 || hidden < 1) return 1;
    double *q = malloc(sizeof(double) * (size_t)dh);
    double *k = malloc(sizeof(double) * (size_t)dh);
    double *h = malloc(sizeof(double) * (size_t)hidden);
    if (!q || !k || !h) { free(q); free(k); free(h); return 2; }
    for (int i = 0; i < n; ++i) {
        feature_map(Xq + (long)i * dh, q, dh, relu_inputs);
        feature_map(Xk + (long)i * dh, k, dh, relu_inputs);
        mlp_step_weights(q, k, dh, T, W1, b1, W2, b2, hidden, h, out + (long)i * T);
    }
    free(q); free(k); free(h);
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int lisa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
