"""Pins of the double-precision oracle against what the LiSA method fixes.

Each test checks the oracle against something other than itself: exact
fractions worked by hand, closed forms, invariants the method guarantees
(row-stochastic, rank <= d_h, T = 1 identity, constant-V preservation, the
untruncated series and its tail), special cases that reduce to a textbook
formula (linear attention, box mean), and a second evaluation route
(explicit n x n walk vs the low-rank recurrence).

Source: "LiSA: Linear Stochastic Attention for Long-Range Visual Modeling"
(reading note of arXiv 2611.04216v2), sections 2.1-2.5.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _rand(B, heads, n, d, scale=1.0):
    return scale * RNG.standard_normal((B, heads, n, d))


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _frac(s):
    return float(Fraction(s))


# -- walk weights (paper Eq. 4) ------------------------------------------------

def test_geometric_weights_golden():
    for row in _golden_rows("geometric_weights.txt"):
        beta, T = float(row[0]), int(row[1])
        want = np.array([_frac(x) for x in row[2:]])
        got = oracle.geometric_weights(beta, T)
        assert got.shape == (T,)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)
        assert abs(got.sum() - 1.0) < 1e-15


def test_geometric_weights_reject_bad_args():
    for beta, T in ((1.0, 3), (-0.1, 3), (0.5, 0)):
        with pytest.raises(ValueError):
            oracle.geometric_weights(beta, T)


# -- hand-worked examples ------------------------------------------------------

def test_worked_example_global_branch():
    row = [r for r in _golden_rows("worked_examples.txt") if r[0] == "global_1x2"][0]
    want = np.array([_frac(x) for x in row[2:]])
    q = np.array([1.0, 1.0]).reshape(1, 1, 2, 1)
    k = np.array([1.0, 3.0]).reshape(1, 1, 2, 1)
    v = np.array([0.0, 4.0]).reshape(1, 1, 2, 1)
    for mode in (oracle.EXPLICIT, oracle.LOWRANK):
        _, G, _ = oracle.forward(q, k, v, (1, 2), 3, alpha=1.0, beta=0.5, eps=0.0, mode=mode,
                                 branches=True)
        np.testing.assert_allclose(G.reshape(-1), want, rtol=1e-14)


def test_worked_example_local_branch():
    row = [r for r in _golden_rows("worked_examples.txt") if r[0] == "local_1x2"][0]
    want = np.array([_frac(x) for x in row[2:]])
    q = np.zeros((1, 1, 2, 4)); q[0, 0, 0, 0] = 1.0; q[0, 0, 1, 0] = 2.0
    k = np.zeros((1, 1, 2, 4)); k[0, 0, 1, 0] = 2.0 * math.log(3.0)
    v = np.array([1.0, 5.0]).reshape(1, 1, 2, 1)
    _, _, L = oracle.forward(q, k, v, (1, 2), 3, alpha=0.0, beta=0.5, branches=True)
    np.testing.assert_allclose(L.reshape(-1), want, rtol=1e-14)


# -- the transition matrix (note section 2.2) -----------------------------------

@pytest.mark.parametrize("grid,d", [((14, 14), 16), ((4, 5), 8), ((1, 7), 3)])
def test_transition_row_stochastic_and_low_rank(grid, d):
    n = grid[0] * grid[1]
    xq, xk = RNG.standard_normal((n, d)), RNG.standard_normal((n, d))
    S = oracle.transition(xq, xk, eps=1e-6)
    assert (S >= 0).all()
    # rows sum to 1 up to the stabiliser: 1 - sum_j S_ij = eps / (Q_i . s + eps)
    S0 = oracle.transition(xq, xk, eps=0.0)
    live = np.abs(S0.sum(1)) > 0            # a query row that ReLU zeroed stays zero
    np.testing.assert_allclose(S0.sum(1)[live], 1.0, rtol=0, atol=1e-13)
    assert (S.sum(1) <= 1.0 + 1e-13).all()
    assert (S.sum(1)[live] > 1.0 - 1e-5).all()
    # rank at most d_h: product of an n x d_h and a d_h x n factor
    sv = np.linalg.svd(S, compute_uv=False)
    if n > d:
        assert sv[d] <= 1e-12 * sv[0]


# -- two evaluation routes agree (note section 2.3) -------------------------------

@pytest.mark.parametrize("grid,d,T", [((1, 1), 4, 3), ((1, 5), 4, 4), ((3, 3), 8, 5),
                                      ((4, 5), 16, 3), ((14, 14), 16, 3), ((7, 9), 8, 1)])
def test_explicit_matches_lowrank(grid, d, T):
    n = grid[0] * grid[1]
    xq, xk, v = _rand(2, 2, n, d), _rand(2, 2, n, d), _rand(2, 2, n, d)
    alpha = np.array([0.3, 0.8])
    a = oracle.forward(xq, xk, v, grid, T, alpha=alpha, beta=0.5, mode=oracle.EXPLICIT)
    b = oracle.forward(xq, xk, v, grid, T, alpha=alpha, beta=0.5, mode=oracle.LOWRANK)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-10 * np.abs(a).max())


def test_explicit_matches_lowrank_mlp():
    grid, d, T, hid = (5, 6), 8, 4, 7
    n = 30
    xq, xk, v = _rand(1, 3, n, d), _rand(1, 3, n, d), _rand(1, 3, n, d)
    mlp = (0.5 * RNG.standard_normal((hid, 2 * d)), 0.5 * RNG.standard_normal(hid),
           0.5 * RNG.standard_normal((T, hid)), 0.5 * RNG.standard_normal(T))
    a = oracle.forward(xq, xk, v, grid, T, alpha=0.5, mlp=mlp, mode=oracle.EXPLICIT)
    b = oracle.forward(xq, xk, v, grid, T, alpha=0.5, mlp=mlp, mode=oracle.LOWRANK)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-10 * np.abs(a).max())


@pytest.mark.parametrize("grid", [(1, 1), (1, 5), (3, 3), (4, 5)])
@pytest.mark.parametrize("k", [0, 1, 2, 3])
def test_single_hop_term_is_matrix_power(grid, k):
    """Fixed weights w = e_k isolate S^k V; compare with a dense power of S."""
    n, d, T = grid[0] * grid[1], 4, 4
    xq, xk, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, d)
    w = np.zeros(T); w[k] = 1.0
    S = oracle.transition(xq[0, 0], xk[0, 0], eps=1e-6)
    want = np.linalg.matrix_power(S, k) @ v[0, 0]
    for mode in (oracle.EXPLICIT, oracle.LOWRANK):
        _, G, _ = oracle.forward(xq, xk, v, grid, T, alpha=1.0, w=w, mode=mode, branches=True)
        np.testing.assert_allclose(G[0, 0], want, rtol=1e-11, atol=1e-12)


# -- special cases the pages fix ---------------------------------------------------

def test_T1_global_is_V_exactly():
    """T = 1 keeps only the S^0 = I self-loop (note section 2.2)."""
    xq, xk, v = _rand(2, 2, 12, 4), _rand(2, 2, 12, 4), _rand(2, 2, 12, 4)
    for mode in (oracle.EXPLICIT, oracle.LOWRANK):
        _, G, _ = oracle.forward(xq, xk, v, (3, 4), 1, alpha=1.0, beta=0.5, mode=mode, branches=True)
        assert np.array_equal(G, v)


def test_constant_V_is_preserved():
    """P is row-stochastic, so a constant value field passes through both
    branches; the stabiliser eps only shrinks the hop terms by ~eps."""
    n, d = 20, 8
    xq, xk = _rand(1, 2, n, d), _rand(1, 2, n, d)
    v = np.full((1, 2, n, d), 2.5)
    O, G, L = oracle.forward(xq, xk, v, (4, 5), 5, alpha=[0.25, 0.75], beta=0.5, branches=True)
    np.testing.assert_allclose(L, 2.5, rtol=1e-14)
    np.testing.assert_allclose(G, 2.5, rtol=1e-6)
    np.testing.assert_allclose(O, 2.5, rtol=1e-6)
    O0, G0, _ = oracle.forward(xq, xk, v, (4, 5), 5, alpha=0.5, beta=0.5, eps=0.0, branches=True)
    np.testing.assert_allclose(G0, 2.5, rtol=1e-13)


def test_linear_attention_special_case():
    """w = (0, 1) gives S V = Q~ K^T V: normalised kernel linear attention with
    the ReLU feature map (paper Eq. 3)."""
    n, d, dv = 24, 6, 5
    xq, xk, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, dv)
    eps = 1e-3
    _, G, _ = oracle.forward(xq, xk, v, (4, 6), 2, alpha=1.0, w=[0.0, 1.0], eps=eps, branches=True)
    phq, phk = np.maximum(xq[0, 0], 0), np.maximum(xk[0, 0], 0)
    want = (phq @ (phk.T @ v[0, 0])) / (phq @ phk.sum(0) + eps)[:, None]
    np.testing.assert_allclose(G[0, 0], want, rtol=1e-12)


@pytest.mark.parametrize("beta", [0.3, 0.5, 0.8])
def test_untruncated_closed_form(beta):
    """As T grows the truncated walk tends to (1-beta)(I - beta S)^-1 V
    (note section 2.3), and the gap shrinks monotonically."""
    grid, d = (3, 4), 5
    n = 12
    xq, xk, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, 3)
    S = oracle.transition(xq[0, 0], xk[0, 0], eps=1e-6)
    closed = (1 - beta) * np.linalg.solve(np.eye(n) - beta * S, v[0, 0])
    gaps = []
    for T in (2, 4, 8, 16, 140):
        _, G, _ = oracle.forward(xq, xk, v, grid, T, alpha=1.0, beta=beta, branches=True)
        gaps.append(np.abs(G[0, 0] - closed).max())
    assert all(b < a for a, b in zip(gaps, gaps[1:-1]))
    assert gaps[-1] < 1e-12


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_truncation_tail_norm(T):
    """With S exactly row-stochastic (eps = 0) the dropped tail
    R_T = (1-beta) sum_{k >= T} beta^k S^k has entrywise l1 norm n beta^T
    (note section 2.5, paper Supp. Sec. 6).  The bound is about the
    unnormalised tail, not about the renormalised truncation."""
    beta, n = 0.5, 9
    xq, xk = np.abs(RNG.standard_normal((n, 4))) + 0.1, np.abs(RNG.standard_normal((n, 4))) + 0.1
    S = oracle.transition(xq, xk, eps=0.0)
    full = (1 - beta) * np.linalg.inv(np.eye(n) - beta * S)
    part = sum((1 - beta) * beta ** k * np.linalg.matrix_power(S, k) for k in range(T))
    R = full - part
    assert (R >= -1e-15).all()
    assert abs(np.abs(R).sum() - n * beta ** T) <= 1e-9 * n


# -- untruncated walk (T = 0): (1-beta)(I - beta S)^-1 V, note section 2.3 -----------

@pytest.mark.parametrize("beta", [0.0, 0.3, 0.5, 0.9])
def test_untruncated_routes_agree_with_library_solve(beta):
    """The oracle's two untruncated routes (dense n x n elimination, and the
    d x d push-through solve) against LAPACK's solve of the n x n system."""
    grid, d, n = (4, 5), 6, 20
    xq, xk, v = _rand(2, 1, n, d), _rand(2, 1, n, d), _rand(2, 1, n, 7)
    _, Ge, _ = oracle.forward(xq, xk, v, grid, 0, alpha=1.0, beta=beta, mode=oracle.EXPLICIT, branches=True)
    _, Gl, _ = oracle.forward(xq, xk, v, grid, 0, alpha=1.0, beta=beta, mode=oracle.LOWRANK, branches=True)
    for b in range(2):
        S = oracle.transition(xq[b, 0], xk[b, 0], eps=1e-6)
        want = (1 - beta) * np.linalg.solve(np.eye(n) - beta * S, v[b, 0])
        np.testing.assert_allclose(Ge[b, 0], want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(Gl[b, 0], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("beta", [0.25, 0.5, 0.8])
def test_untruncated_is_limit_of_truncated_series(beta):
    """The untruncated walk is the T -> infinity limit of the renormalised
    truncated one (paper Eq. 4 with 1 - beta^T -> 1), reached through the
    independently pinned power-series route; the gap falls like beta^T."""
    grid, d, n = (6, 6), 8, 36
    xq, xk, v = _rand(1, 2, n, d), _rand(1, 2, n, d), _rand(1, 2, n, d)
    _, Ginf, _ = oracle.forward(xq, xk, v, grid, 0, alpha=1.0, beta=beta, branches=True)
    gaps = []
    for T in (2, 4, 8, 16):
        _, G, _ = oracle.forward(xq, xk, v, grid, T, alpha=1.0, beta=beta, branches=True)
        gaps.append(np.abs(G - Ginf).max())
    assert all(b < a for a, b in zip(gaps, gaps[1:]))
    _, Gfar, _ = oracle.forward(xq, xk, v, grid, 200, alpha=1.0, beta=beta, branches=True)
    assert np.abs(Gfar - Ginf).max() < 1e-11


@pytest.mark.parametrize("T", [1, 2, 4, 7])
def test_untruncated_tail_norm_through_the_oracle(T):
    """With eps = 0 (S exactly row-stochastic), V = I_n makes the global branch
    the walk matrix itself: the untruncated P minus the unnormalised truncated
    sum (1-beta) beta^k S^k, k < T, is the tail R_T with entrywise l1 norm
    n beta^T (note section 2.5, paper Supp. Sec. 6)."""
    beta, n, grid = 0.5, 12, (3, 4)
    xq = np.abs(RNG.standard_normal((1, 1, n, 5))) + 0.1
    xk = np.abs(RNG.standard_normal((1, 1, n, 5))) + 0.1
    eye = np.eye(n)[None, None]
    _, P, _ = oracle.forward(xq, xk, eye, grid, 0, alpha=1.0, beta=beta, eps=0.0, branches=True)
    w = (1 - beta) * beta ** np.arange(T)
    _, PT, _ = oracle.forward(xq, xk, eye, grid, T, alpha=1.0, w=w, eps=0.0, branches=True)
    R = P[0, 0] - PT[0, 0]
    assert (R >= -1e-14).all()
    assert abs(np.abs(R).sum() - n * beta ** T) <= 1e-9 * n
    np.testing.assert_allclose(P[0, 0].sum(axis=1), 1.0, rtol=0, atol=1e-12)   # P row-stochastic


def test_untruncated_special_values():
    """beta = 0 keeps only the self-loop (g = V); a constant value field is
    preserved (P row-stochastic up to eps); a zero query row gets (1-beta) V_i."""
    grid, n, d = (3, 5), 15, 6
    xq, xk, v = _rand(1, 1, n, d), _rand(1, 1, n, d), _rand(1, 1, n, d)
    _, G, _ = oracle.forward(xq, xk, v, grid, 0, alpha=1.0, beta=0.0, branches=True)
    assert np.array_equal(G, v)
    c = np.full((1, 1, n, d), -1.75)
    for mode in (oracle.EXPLICIT, oracle.LOWRANK):
        _, G, _ = oracle.forward(xq, xk, c, grid, 0, alpha=1.0, beta=0.7, eps=0.0, mode=mode, branches=True)
        np.testing.assert_allclose(G, -1.75, rtol=1e-13)
    xz = xq.copy()
    xz[0, 0, 4] = -1.0     # ReLU'd to a zero query row: Q~_4 = 0
    _, G, _ = oracle.forward(xz, xk, v, grid, 0, alpha=1.0, beta=0.6, branches=True)
    np.testing.assert_allclose(G[0, 0, 4], 0.4 * v[0, 0, 4], rtol=1e-14)


def test_untruncated_rejects_non_geometric_weights():
    xq = _rand(1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.forward(xq, xq, xq, (2, 2), 0, alpha=1.0, w=[1.0])
    with pytest.raises(ValueError):
        oracle.forward(xq, xq, xq, (2, 2), 0, alpha=1.0, beta=1.0)


# -- local branch (note section 2.4) -------------------------------------------------

def _box_mean(v, H, W):
    out = np.zeros_like(v)
    for r in range(H):
        for c in range(W):
            rs = slice(max(r - 1, 0), min(r + 2, H))
            cs = slice(max(c - 1, 0), min(c + 2, W))
            out[r * W + c] = v.reshape(H, W, -1)[rs, cs].reshape(-1, v.shape[-1]).mean(0)
    return out


@pytest.mark.parametrize("grid", [(1, 1), (1, 6), (5, 1), (4, 7), (6, 6)])
def test_local_zero_query_is_box_mean(grid):
    """All scores zero -> uniform weights over the in-grid window: 1/4 at
    corners, 1/6 on edges, 1/9 inside (neighbours outside are left out)."""
    H, W = grid
    n, d = H * W, 4
    xq = -np.abs(_rand(1, 1, n, d)) - 0.1          # ReLU -> Q = 0
    xk, v = _rand(1, 1, n, d), _rand(1, 1, n, 3)
    O, G, L = oracle.forward(xq, xk, v, grid, 3, alpha=0.4, beta=0.5, branches=True)
    box = _box_mean(v[0, 0], H, W)
    np.testing.assert_allclose(L[0, 0], box, rtol=1e-13, atol=1e-14)
    w0 = oracle.geometric_weights(0.5, 3)[0]
    np.testing.assert_allclose(G[0, 0], w0 * v[0, 0], rtol=1e-14)   # Q~ = 0
    np.testing.assert_allclose(O[0, 0], 0.4 * w0 * v[0, 0] + 0.6 * box, rtol=1e-12, atol=1e-14)
    if n > 1:
        counts = np.array([[(min(r + 2, H) - max(r - 1, 0)) * (min(c + 2, W) - max(c - 1, 0))
                            for c in range(W)] for r in range(H)])
        assert counts.max() <= 9 and counts.min() >= (2 if min(H, W) == 1 else 4)


def test_local_single_marked_key_non_square():
    """One key carries a large code; queries all read it.  For i in the window
    of p the weight on p is e^a / (e^a + |N(i)| - 1), a = c/sqrt(d_h); tokens
    outside that window see uniform weights.  Non-square grid catches a swap
    of rows and columns; the weight catches a wrong scale or a transposed
    score (q_j . k_i instead of q_i . k_j)."""
    H, W, d, cval = 5, 7, 16, 6.0
    n = H * W
    p = 2 * W + 5
    xq = np.zeros((1, 1, n, d)); xq[..., 0] = 1.0
    xk = np.zeros((1, 1, n, d)); xk[0, 0, p, 0] = cval
    v = np.zeros((1, 1, n, 1)); v[0, 0, p, 0] = 1.0
    _, _, L = oracle.forward(xq, xk, v, (H, W), 3, alpha=0.0, beta=0.5, branches=True)
    a = math.exp(cval / math.sqrt(d))
    pr, pc = divmod(p, W)
    for i in range(n):
        r, c = divmod(i, W)
        cnt = (min(r + 2, H) - max(r - 1, 0)) * (min(c + 2, W) - max(c - 1, 0))
        near = abs(r - pr) <= 1 and abs(c - pc) <= 1
        want = a / (a + cnt - 1) if near else 0.0
        assert abs(L[0, 0, i, 0] - want) < 1e-14, (i, L[0, 0, i, 0], want)


def test_local_one_by_one_grid_returns_V():
    xq, xk, v = _rand(1, 2, 1, 8), _rand(1, 2, 1, 8), _rand(1, 2, 1, 8)
    _, _, L = oracle.forward(xq, xk, v, (1, 1), 3, alpha=0.5, beta=0.5, branches=True)
    np.testing.assert_allclose(L, v, rtol=1e-15)


# -- adaptive weights (note section 2.4, paper Eq. 10) ----------------------------------

def test_mlp_reduces_to_geometric():
    """W1 = W2 = 0 and b2 = log w_geo give softmax(log w_geo) = w_geo."""
    d, T, hid = 8, 4, 5
    xq, xk, v = _rand(2, 2, 15, d), _rand(2, 2, 15, d), _rand(2, 2, 15, d)
    wg = oracle.geometric_weights(0.5, T)
    mlp = (np.zeros((hid, 2 * d)), RNG.standard_normal(hid), np.zeros((T, hid)), np.log(wg))
    a = oracle.forward(xq, xk, v, (3, 5), T, alpha=[0.2, 0.9], mlp=mlp)
    b = oracle.forward(xq, xk, v, (3, 5), T, alpha=[0.2, 0.9], beta=0.5)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    mlp0 = (np.zeros((hid, 2 * d)), np.zeros(hid), np.zeros((T, hid)), np.zeros(T))
    c = oracle.forward(xq, xk, v, (3, 5), T, alpha=[0.2, 0.9], mlp=mlp0)
    e = oracle.forward(xq, xk, v, (3, 5), T, alpha=[0.2, 0.9], w=np.full(T, 1.0 / T))
    np.testing.assert_allclose(c, e, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("col", [1, 8 + 2])
def test_mlp_single_path_closed_form(col):
    """One hidden unit reading one input coordinate: z_1 = GELU(x_col + b) with
    the exact erf GELU, x = concat(q, k) (q first).  The weights are a
    3-way softmax of (b2_0, z_1 + b2_1, b2_2)."""
    d, T, hid, n = 8, 3, 4, 10
    xq, xk = RNG.standard_normal((n, d)), RNG.standard_normal((n, d))
    W1 = np.zeros((hid, 2 * d)); W1[0, col] = 1.0
    b1 = np.array([0.1, 0.0, 0.0, 0.0])
    W2 = np.zeros((T, hid)); W2[1, 0] = 1.0
    b2 = np.array([0.05, -0.2, 0.3])
    got = oracle.step_weights(xq, xk, (W1, b1, W2, b2), T)
    x = np.concatenate([np.maximum(xq, 0), np.maximum(xk, 0)], axis=1)[:, col]
    pre = x + 0.1
    gelu = 0.5 * pre * (1 + np.array([math.erf(t / math.sqrt(2)) for t in pre]))
    z = np.stack([np.full(n, b2[0]), gelu + b2[1], np.full(n, b2[2])], axis=1)
    want = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    np.testing.assert_allclose(got, want, rtol=1e-14)


# -- mixing, slicing and feature map ------------------------------------------------

def test_alpha_selects_branches_per_head():
    xq, xk, v = _rand(2, 3, 20, 4), _rand(2, 3, 20, 4), _rand(2, 3, 20, 4)
    alpha = np.array([1.0, 0.0, 0.3])
    O, G, L = oracle.forward(xq, xk, v, (4, 5), 3, alpha=alpha, beta=0.5, branches=True)
    assert np.array_equal(O[:, 0], G[:, 0])
    assert np.array_equal(O[:, 1], L[:, 1])
    np.testing.assert_allclose(O[:, 2], 0.3 * G[:, 2] + 0.7 * L[:, 2], rtol=1e-15)


def test_slices_are_independent_and_relu_flag():
    xq, xk, v = _rand(3, 2, 12, 4), _rand(3, 2, 12, 4), _rand(3, 2, 12, 4)
    full = oracle.forward(xq, xk, v, (3, 4), 3, alpha=[0.5, 0.6], beta=0.5)
    one = oracle.forward(xq[1:2, 1:2], xk[1:2, 1:2], v[1:2, 1:2], (3, 4), 3, alpha=[0.6], beta=0.5)
    assert np.array_equal(full[1, 1], one[0, 0])
    pre = oracle.forward(np.maximum(xq, 0), np.maximum(xk, 0), v, (3, 4), 3, alpha=[0.5, 0.6],
                         beta=0.5, relu=False)
    assert np.array_equal(full, pre)


def test_zero_query_row_gives_w0_V():
    """A query row that ReLU zeroes has Q~_i = 0 and g_i = w_0 V_i."""
    xq, xk, v = _rand(1, 1, 12, 4), _rand(1, 1, 12, 4), _rand(1, 1, 12, 4)
    xq[0, 0, 5] = -1.0
    _, G, _ = oracle.forward(xq, xk, v, (3, 4), 3, alpha=1.0, beta=0.5, branches=True)
    w0 = oracle.geometric_weights(0.5, 3)[0]
    assert G[0, 0, 5].tolist() == (w0 * v[0, 0, 5]).tolist()


# -- the ELU + 1 feature map (note section 2.1; paper Table 8 compares ELU with ReLU) -------

def test_elu_feature_map_transition_is_row_stochastic_and_low_rank():
    """phi(x) = ELU(x) + 1 > 0 keeps S non-negative with rows summing to
    Q~_i . s < 1 by eps only, and of rank <= d_h, like the ReLU map."""
    n, d = 30, 4
    xq, xk = RNG.standard_normal((n, d)), RNG.standard_normal((n, d))
    S = oracle.transition(xq, xk, eps=1e-6, relu="elu1")
    assert (S > 0).all()                                   # every feature positive: no zero entries
    np.testing.assert_allclose(S.sum(axis=1), 1.0, rtol=0, atol=1e-5)
    assert np.linalg.matrix_rank(S, tol=1e-10) <= d
    S0 = oracle.transition(xq, xk, eps=0.0, relu="elu1")
    np.testing.assert_allclose(S0.sum(axis=1), 1.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("T", [0, 1, 3, 5])
def test_elu_feature_map_routes_agree(T):
    grid, d = (4, 5), 6
    xq, xk, v = _rand(1, 2, 20, d), _rand(1, 2, 20, d), _rand(1, 2, 20, d)
    e = oracle.forward(xq, xk, v, grid, T, alpha=[0.4, 0.6], beta=0.5, relu="elu1", mode=oracle.EXPLICIT)
    l = oracle.forward(xq, xk, v, grid, T, alpha=[0.4, 0.6], beta=0.5, relu="elu1", mode=oracle.LOWRANK)
    np.testing.assert_allclose(e, l, rtol=0, atol=1e-10)


def test_elu_feature_map_differs_from_relu_and_matches_on_positive_inputs_shifted():
    """For inputs all > 0, ELU(x) + 1 = x + 1: the ELU layer on X equals the
    no-feature-map layer on X + 1 (a closed form of the map)."""
    grid, d = (3, 4), 5
    xq, xk, v = np.abs(_rand(1, 1, 12, d)) + 0.1, np.abs(_rand(1, 1, 12, d)) + 0.1, _rand(1, 1, 12, d)
    a = oracle.forward(xq, xk, v, grid, 3, alpha=0.5, beta=0.5, relu="elu1")
    b = oracle.forward(xq + 1.0, xk + 1.0, v, grid, 3, alpha=0.5, beta=0.5, relu=False)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    c = oracle.forward(xq, xk, v, grid, 3, alpha=0.5, beta=0.5, relu=True)
    assert np.abs(a - c).max() > 1e-3


def test_feature_map_argument_checked():
    xq = _rand(1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.forward(xq, xq, xq, (2, 2), 3, alpha=0.5, beta=0.5, relu="elu")
