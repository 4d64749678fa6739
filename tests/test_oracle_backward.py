"""Pins of the oracle's backward pass (dL/dXq, dL/dXk, dL/dV, dL/dalpha).

The oracle's backward is the chain rule written out by hand through the
forward's steps.  It is checked against routes that share nothing with that
derivation: central finite differences of the (separately pinned) forward,
and torch autograd through a dense n x n restatement of the layer (S formed,
walk powers S^k V, the 3x3 window as a masked softmax).  Plus closed forms:
T = 1 with alpha = 1 makes the layer the identity on V, and the gradient is
linear in the upstream gradient.

Source: "LiSA: Linear Stochastic Attention for Long-Range Visual Modeling"
(reading note of arXiv 2611.04216v2), sections 2.1-2.5.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(4321)


def _case(B, heads, H, W, d, scale=1.0):
    n = H * W
    return [scale * RNG.standard_normal((B, heads, n, d)) for _ in range(4)]


def _loss(xq, xk, v, dO, grid, T, alpha, **kw):
    return float((oracle.forward(xq, xk, v, grid, T, alpha=alpha, **kw) * dO).sum())


WEIGHTS = [(3, {"beta": 0.5}), (4, {"w": [0.2, -0.5, 1.3, 0.7]}), (1, {"beta": 0.5}), (0, {"beta": 0.6}),
           (6, {"beta": 0.8})]


@pytest.mark.parametrize("T,kw", WEIGHTS)
@pytest.mark.parametrize("grid", [(3, 4), (1, 5), (4, 1)])
def test_backward_matches_finite_differences(T, kw, grid):
    H, W = grid
    xq, xk, v, dO = _case(1, 2, H, W, 5)
    alpha = np.array([0.3, 0.7])
    gq, gk, gv, ga = oracle.backward(xq, xk, v, dO, grid, T, alpha=alpha, **kw)
    h = 1e-6
    for arr, grad in ((xq, gq), (xk, gk), (v, gv)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + h
            up = _loss(xq, xk, v, dO, grid, T, alpha, **kw)
            arr[idx] = keep - h
            dn = _loss(xq, xk, v, dO, grid, T, alpha, **kw)
            arr[idx] = keep
            num[idx] = (up - dn) / (2 * h)
        assert np.abs(num - grad).max() <= 1e-6 * max(np.abs(grad).max(), 1.0)
    for hd in range(2):
        e = np.zeros(2)
        e[hd] = h
        num = (_loss(xq, xk, v, dO, grid, T, alpha + e, **kw) - _loss(xq, xk, v, dO, grid, T, alpha - e, **kw)) / (2 * h)
        assert abs(num - ga[hd]) <= 1e-6 * max(abs(ga[hd]), 1.0)


def test_backward_without_feature_map():
    """relu = False: the inputs are the (non-negative) features themselves."""
    xq, xk, v, dO = _case(1, 1, 3, 3, 4)
    xq, xk = np.abs(xq) + 0.05, np.abs(xk) + 0.05
    grid, T = (3, 3), 3
    gq, gk, gv, _ = oracle.backward(xq, xk, v, dO, grid, T, alpha=0.4, beta=0.5, relu=False)
    h = 1e-6
    for arr, grad in ((xq, gq), (xk, gk)):
        for idx in [(0, 0, 0, 0), (0, 0, 4, 2), (0, 0, 8, 3)]:
            keep = arr[idx]
            arr[idx] = keep + h
            up = _loss(xq, xk, v, dO, grid, T, 0.4, beta=0.5, relu=False)
            arr[idx] = keep - h
            dn = _loss(xq, xk, v, dO, grid, T, 0.4, beta=0.5, relu=False)
            arr[idx] = keep
            assert abs((up - dn) / (2 * h) - grad[idx]) <= 1e-6 * max(abs(grad[idx]), 1.0)


def _dense_torch_layer(xq, xk, v, grid, T, alpha, w, eps=1e-6):
    """The layer restated densely in torch (autograd's route): S = Q~ K^T
    formed, g = sum_k w_k S^k V, the local window as a masked softmax."""
    H, W = grid
    n = H * W
    q, k = torch.relu(xq), torch.relu(xk)
    s = k.sum(0)
    qt = q / (q @ s + eps)[:, None]
    S = qt @ k.T
    g, y = w[0] * v, v
    for t in range(1, T):
        y = S @ y
        g = g + w[t] * y
    rr, cc = np.divmod(np.arange(n), W)
    near = (np.abs(rr[:, None] - rr[None, :]) <= 1) & (np.abs(cc[:, None] - cc[None, :]) <= 1)
    e = (q @ k.T) / np.sqrt(q.shape[1])
    e = e.masked_fill(torch.from_numpy(~near), float("-inf"))
    l = torch.softmax(e, dim=1) @ v
    return alpha * g + (1 - alpha) * l


@pytest.mark.parametrize("T,w", [(3, [4 / 7, 2 / 7, 1 / 7]), (4, [0.1, 0.4, -0.3, 0.8])])
def test_backward_matches_autograd_of_dense_layer(T, w):
    grid = (5, 4)
    xq, xk, v, dO = _case(1, 1, 5, 4, 6)
    alpha = 0.35
    gq, gk, gv, ga = oracle.backward(xq, xk, v, dO, grid, T, alpha=alpha, w=w)
    t = [torch.tensor(a[0, 0], requires_grad=True) for a in (xq, xk, v)]
    ta = torch.tensor(alpha, dtype=torch.float64, requires_grad=True)
    out = _dense_torch_layer(t[0], t[1], t[2], grid, T, ta, w)
    np.testing.assert_allclose(out.detach().numpy(), oracle.forward(xq, xk, v, grid, T, alpha=alpha, w=w)[0, 0],
                               rtol=0, atol=1e-12)
    (out * torch.from_numpy(dO[0, 0])).sum().backward()
    for got, ref in ((gq, t[0]), (gk, t[1]), (gv, t[2])):
        np.testing.assert_allclose(got[0, 0], ref.grad.numpy(), rtol=0, atol=1e-10)
    assert abs(ga[0] - ta.grad.item()) <= 1e-10


def test_identity_layer_gradients():
    """T = 1, alpha = 1: O = V exactly, so dXq = dXk = 0, dV = dO, and
    dalpha = sum dO . (V - l) (the local branch still enters through alpha)."""
    xq, xk, v, dO = _case(2, 1, 4, 3, 4)
    gq, gk, gv, ga = oracle.backward(xq, xk, v, dO, (4, 3), 1, alpha=1.0, beta=0.5)
    assert np.all(gq == 0) and np.all(gk == 0)
    np.testing.assert_allclose(gv, dO, rtol=0, atol=1e-15)
    _, _, L = oracle.forward(xq, xk, v, (4, 3), 1, alpha=1.0, beta=0.5, branches=True)
    np.testing.assert_allclose(ga[0], (dO * (v - L)).sum(), rtol=1e-13)


def test_backward_is_linear_in_upstream_gradient():
    xq, xk, v, d1 = _case(1, 2, 3, 5, 4)
    d2 = RNG.standard_normal(d1.shape)
    kw = dict(alpha=[0.2, 0.6], beta=0.5)
    a = oracle.backward(xq, xk, v, d1, (3, 5), 3, **kw)
    b = oracle.backward(xq, xk, v, d2, (3, 5), 3, **kw)
    c = oracle.backward(xq, xk, v, d1 + 2 * d2, (3, 5), 3, **kw)
    for x, y, z in zip(a, b, c):
        np.testing.assert_allclose(z, x + 2 * y, rtol=1e-12, atol=1e-12)


def test_backward_rejects_mlp_and_bad_args():
    xq, xk, v, dO = _case(1, 1, 2, 2, 3)
    with pytest.raises(ValueError):
        oracle.backward(xq, xk, v, dO, (2, 2), 0, alpha=0.5, w=[1.0])
    with pytest.raises(ValueError):
        oracle.backward(xq, xk, v, dO, (2, 3), 3, alpha=0.5, beta=0.5)


# -- adaptive (MLP) walk weights (note section 2.4; paper Eq. 10, Supp. Sec. 8) ----------

def _mlp_params(d, T, hidden=6, seed=5):
    r = np.random.default_rng(seed)
    return (0.4 * r.standard_normal((hidden, 2 * d)), 0.3 * r.standard_normal(hidden),
            0.5 * r.standard_normal((T, hidden)), 0.2 * r.standard_normal(T))


@pytest.mark.parametrize("T", [1, 3, 4])
def test_mlp_backward_matches_finite_differences(T):
    grid, d = (3, 4), 5
    xq, xk, v, dO = _case(1, 2, 3, 4, d)
    mlp = _mlp_params(d, T)
    alpha = np.array([0.3, 0.7])
    gq, gk, gv, ga, gp = oracle.backward(xq, xk, v, dO, grid, T, alpha=alpha, mlp=mlp)
    args = [xq, xk, v, alpha] + [np.array(x) for x in mlp]
    grads = [gq, gk, gv, ga] + list(gp)

    def loss():
        return float((oracle.forward(args[0], args[1], args[2], grid, T, alpha=args[3],
                                     mlp=tuple(args[4:])) * dO).sum())
    h = 1e-6
    for arr, grad in zip(args, grads):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + h
            up = loss()
            arr[idx] = keep - h
            dn = loss()
            arr[idx] = keep
            num[idx] = (up - dn) / (2 * h)
        assert np.abs(num - grad).max() <= 1e-6 * max(np.abs(grad).max(), 1.0)


def test_mlp_backward_matches_autograd_of_dense_layer():
    grid, T, d = (4, 4), 3, 4
    xq, xk, v, dO = _case(1, 1, 4, 4, d)
    W1, b1, W2, b2 = _mlp_params(d, T, hidden=5, seed=9)
    alpha = 0.6
    gq, gk, gv, ga, (gW1, gb1, gW2, gb2) = oracle.backward(xq, xk, v, dO, grid, T, alpha=alpha,
                                                           mlp=(W1, b1, W2, b2))
    t = [torch.tensor(a[0, 0], requires_grad=True) for a in (xq, xk, v)]
    tp = [torch.tensor(p, requires_grad=True) for p in (W1, b1, W2, b2)]
    ta = torch.tensor(alpha, dtype=torch.float64, requires_grad=True)
    q, k = torch.relu(t[0]), torch.relu(t[1])
    hdn = torch.nn.functional.gelu(torch.cat([q, k], 1) @ tp[0].T + tp[1])   # exact erf GELU
    w = torch.softmax(hdn @ tp[2].T + tp[3], dim=1)                          # [n, T]
    s = k.sum(0)
    qt = q / (q @ s + 1e-6)[:, None]
    S = qt @ k.T
    y, g = t[2], w[:, :1] * t[2]
    for kk in range(1, T):
        y = S @ y
        g = g + w[:, kk:kk + 1] * y
    n = 16
    rr, cc = np.divmod(np.arange(n), 4)
    near = (np.abs(rr[:, None] - rr[None, :]) <= 1) & (np.abs(cc[:, None] - cc[None, :]) <= 1)
    e = ((q @ k.T) / np.sqrt(d)).masked_fill(torch.from_numpy(~near), float("-inf"))
    out = ta * g + (1 - ta) * (torch.softmax(e, 1) @ t[2])
    (out * torch.from_numpy(dO[0, 0])).sum().backward()
    for got, ref in ((gq, t[0]), (gk, t[1]), (gv, t[2])):
        np.testing.assert_allclose(got[0, 0], ref.grad.numpy(), rtol=0, atol=1e-10)
    for got, ref in zip((gW1, gb1, gW2, gb2), tp):
        np.testing.assert_allclose(got, ref.grad.numpy(), rtol=0, atol=1e-10)
    assert abs(ga[0] - ta.grad.item()) <= 1e-10


def test_mlp_backward_reduces_to_geometric():
    """W2 = 0, b2 = log w_geo: every token gets the geometric weights, so the
    adaptive route (per-token dU_k) gives the geometric backward's feature
    gradients, and the MLP's share of them vanishes (W2^T dz = 0)."""
    grid, T, d = (4, 5), 4, 6
    xq, xk, v, dO = _case(2, 2, 4, 5, d)
    wg = oracle.geometric_weights(0.5, T)
    W1, b1, _, _ = _mlp_params(d, T)
    mlp = (W1, b1, np.zeros((T, W1.shape[0])), np.log(wg))
    a = oracle.backward(xq, xk, v, dO, grid, T, alpha=[0.3, 0.8], mlp=mlp)
    b = oracle.backward(xq, xk, v, dO, grid, T, alpha=[0.3, 0.8], beta=0.5)
    for x, y in zip(a[:4], b):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-12)
    gW1, gb1, gW2, gb2 = a[4]
    assert np.all(gW1 == 0) and np.all(gb1 == 0)
    np.testing.assert_allclose(gb2.sum(), 0.0, atol=1e-12)     # softmax: dz sums to zero per token


@pytest.mark.parametrize("T,kw", [(3, {"beta": 0.5}), (0, {"beta": 0.6}), (3, {"mlp": _mlp_params(5, 3)})])
def test_backward_through_elu_feature_map(T, kw):
    """phi(x) = ELU(x) + 1: the feature map's slope is exp(x) for x <= 0."""
    grid, d = (3, 3), 5
    xq, xk, v, dO = _case(1, 1, 3, 3, d)
    res = oracle.backward(xq, xk, v, dO, grid, T, alpha=0.45, relu="elu1", **kw)
    h = 1e-6
    for arr, grad in ((xq, res[0]), (xk, res[1])):
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + h
            up = float((oracle.forward(xq, xk, v, grid, T, alpha=0.45, relu="elu1", **kw) * dO).sum())
            arr[idx] = keep - h
            dn = float((oracle.forward(xq, xk, v, grid, T, alpha=0.45, relu="elu1", **kw) * dO).sum())
            arr[idx] = keep
            assert abs((up - dn) / (2 * h) - grad[idx]) <= 1e-6 * max(np.abs(grad).max(), 1.0)


# -- how much a wrong walk gradient moves the GPU test cases ---------------------------------

def _walk_gradients(xq, xk, v, dO, w, eps=1e-6, plant=None):
    """The layer at alpha = 1 (the walk alone) restated in the low-rank form
    of the note (section 2.3: S^k V = Q~ M^(k-1) U_1, M = K^T Q~, U_1 = K^T V)
    and differentiated by torch autograd.  `plant` puts a known mistake into
    that backward: "drop_ds" zeroes the gradient reaching s = sum_j K_j,
    "transpose_dM" transposes the one reaching M."""
    xq, xk, v = (torch.tensor(a, requires_grad=True) for a in (xq, xk, v))
    q, k = torch.relu(xq), torch.relu(xk)
    s = k.sum(0)
    if plant == "drop_ds":
        s.register_hook(torch.zeros_like)
    qt = q / (q @ s + eps)[:, None]
    M = k.T @ qt
    if plant == "transpose_dM":
        M.register_hook(lambda g: g.T.contiguous())
    u = k.T @ v
    out = w[0] * v
    for t in range(1, len(w)):
        out = out + w[t] * (qt @ u)
        u = M @ u
    (out * torch.from_numpy(dO)).sum().backward()
    return [a.grad.numpy() for a in (xq, xk, v)]


def test_walk_only_cases_see_a_wrong_walk_gradient():
    """The alpha = 1 cases of the GPU backward tests (same seeded inputs and
    upstream gradient): the restatement above matches the oracle's backward,
    and planting a dropped ds or a transposed dM into it moves dXk or dXq by
    more than five times the bf16 bar (2e-2) of the tensor's own norm in at
    least one case, so a kernel with either mistake fails those tests."""
    from lisa_synth import LayerShape, make_inputs, to_f64
    cases = [(LayerShape("bwd", "bf16", 2, 2, 24, 20, 64, 5, "geometric"), True, 0.9),
             (LayerShape("bwd", "bf16", 2, 2, 9, 12, 64, 5, "geometric"), False, 0.9),
             (LayerShape("bwd", "bf16", 2, 2, 7, 9, 64, 3, "geometric"), False, 0.5)]
    worst = {"drop_ds": 0.0, "transpose_dM": 0.0}
    for shape, structured, beta in cases:
        inp = make_inputs(shape, structured=structured)
        g = torch.Generator("cpu").manual_seed(7)
        dO = to_f64(torch.randn(2, 2, shape.n, shape.d, generator=g).to(torch.bfloat16))
        xq, xk, v = (to_f64(inp[key]) for key in ("xq", "xk", "v"))
        w = oracle.geometric_weights(beta, shape.T)
        ref = oracle.backward(xq, xk, v, dO, (shape.H, shape.W), shape.T, alpha=np.ones(2), beta=beta)
        for b in range(2):
            for h in range(2):
                args = (xq[b, h], xk[b, h], v[b, h], dO[b, h], w)
                want = [r[b, h] for r in ref[:3]]
                for got, r in zip(_walk_gradients(*args), want):
                    assert np.abs(got - r).max() <= 1e-9 * np.abs(r).max()
                for plant in worst:
                    got = _walk_gradients(*args, plant=plant)
                    rel = max(np.abs(x - r).max() / np.abs(r).max() for x, r in zip(got[:2], want[:2]))
                    worst[plant] = max(worst[plant], rel)
    for plant, rel in worst.items():
        assert rel > 5 * 2e-2, (plant, rel)
