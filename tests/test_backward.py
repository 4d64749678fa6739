"""GPU parity of the backward pass (lisa_backward) against the oracle's
hand-derived, finite-difference-pinned backward, on the same seeded inputs
and upstream gradient.

Tolerance: each of dXq, dXk and dV separately, max over (batch, head)
slices of ||gpu - oracle||_inf / ||oracle||_inf of that tensor, <= 1e-4
(fp32) or 2e-2 (bf16 outputs, fp32 arithmetic) -- the forward's bounds;
dalpha (fp32 in both) within 1e-3 relative plus 1e-5 of
sum_i |dO_i| (|g_i| + |l_i|), its own rounding scale.

Only the 1 x 1 grid is measured jointly (each tensor's error against the
largest of the three): there S = Q~K^T = Q.K/(Q.K + eps), so dXq and dXk are
O(eps) differences of O(1) terms and fp32 rounding is as large as they are.

With alpha = 1 the output is the walk alone, so dXq and dXk carry only the
walk's gradient (the reverse recurrence, dM, dU_1 and ds).  On i.i.d. inputs
that gradient is small and a wrong term in it can stay within the bf16 bar;
the alpha = 1 cases therefore include structured inputs (near block-diagonal
S) and deep walks (T = 5, beta = 0.9) on small grids, where a dropped ds or a
transposed dM moves dXq or dXk by 10% or more of its own norm
(test_oracle_backward.py pins that on the CPU)."""
import numpy as np
import pytest
import torch

import oracle
from lisa_synth import SHAPES, LayerShape, make_inputs, to_f64

from helpers import TOL, max_rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa
    build.build()
    lisa.load()


def joint_rel_err(got, want):
    """max over slices of max_t ||got_t - want_t||_inf / max_t ||want_t||_inf."""
    S = got[0].shape[0] * got[0].shape[1]
    num = np.max([np.abs(g - w).reshape(S, -1).max(axis=1) for g, w in zip(got, want)], axis=0)
    den = np.max([np.abs(w).reshape(S, -1).max(axis=1) for w in want], axis=0)
    return float((num / np.where(den > 0, den, 1.0)).max())


def assert_per_tensor(got, want, shape):
    """Each gradient against the oracle on its own norm; the 1 x 1 grid jointly."""
    tol = TOL[shape.dtype]
    if shape.n == 1:
        err = joint_rel_err(got, want)
        assert err <= tol, "1 x 1 grid: joint gradient err %.3e (%s)" % (err, shape.dtype)
        return [err] * 3
    errs = [max_rel_err(g, w) for g, w in zip(got, want)]
    for name, e in zip(("dXq", "dXk", "dV"), errs):
        assert e <= tol, "%s err %.3e > %.0e (%s)" % (name, e, tol, shape.dtype)
    return errs


def _upstream(shape, B, heads, seed=7):
    g = torch.Generator("cpu").manual_seed(seed)
    dO = torch.randn(B, heads, shape.n, shape.d, generator=g)
    return dO.to(torch.bfloat16 if shape.dtype == "bf16" else torch.float32)


def _check(shape, *, B=None, heads=None, beta=0.5, w=None, relu=True, seed=0, structured=False, alpha=None):
    from hop_stochastic_vision_gb300 import lisa
    inp = make_inputs(shape, seed=seed, B=B, heads=heads, structured=structured)
    B, heads = inp["xq"].shape[:2]
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], float(alpha))
    if not relu:
        inp["xq"], inp["xk"] = inp["xq"].clamp_min(0), inp["xk"].clamp_min(0)
    dO = _upstream(shape, B, heads)
    d = to_device(inp)
    kw = {"w": list(w)} if w is not None else {"beta": beta}
    dq, dk, dv, da = lisa.backward(d["xq"], d["xk"], d["v"], dO.cuda(), (shape.H, shape.W), shape.T,
                                   alpha=d["alpha"], relu=relu, **kw)
    torch.cuda.synchronize()
    okw = {"w": np.asarray(w, dtype=np.float64)} if w is not None else {"beta": beta}
    want = oracle.backward(to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"]), to_f64(dO),
                           (shape.H, shape.W), shape.T, alpha=inp["alpha"].double().numpy(), relu=relu, **okw)
    got = [to_f64(x.cpu()) for x in (dq, dk, dv)]
    for g in got:
        assert np.isfinite(g).all()
    errs = assert_per_tensor(got, want[:3], shape)
    # dalpha = sum_i dO_i . (g_i - l_i): its rounding scales with sum |dO| (|g| + |l|)
    _, G, L = oracle.forward(to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"]), (shape.H, shape.W), shape.T,
                             alpha=inp["alpha"].double().numpy(), relu=relu, branches=True, **okw)
    mag = (np.abs(to_f64(dO)) * (np.abs(G) + np.abs(L))).sum(axis=(2, 3)).sum(axis=0)
    da_err = np.abs(da.cpu().double().numpy() - want[3])
    assert (da_err <= 1e-3 * np.abs(want[3]) + 1e-5 * mag).all(), (da_err, want[3], mag)
    return errs


def _shape(dtype, d, H, W, T, B=2, heads=2, alpha="uniform(0.3,0.7)"):
    return LayerShape("bwd", dtype, B, heads, H, W, d, T, "geometric", alpha=alpha)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
def test_widths(dtype, d):
    _check(_shape(dtype, d, 7, 9, 3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_depths(dtype, T):
    _check(_shape(dtype, 32, 11, 10, T))


@pytest.mark.parametrize("T", [1, 2])
def test_short_walks_tensor_path(T):
    """bf16 at d = 64 with T = 1 (no hop term) and T = 2 (no recurrence step):
    the split recurrences' degenerate cases."""
    _check(_shape("bf16", 64, 11, 10, T))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fixed_weights_and_untruncated(dtype):
    _check(_shape(dtype, 64, 9, 12, 4), w=(0.2, -0.5, 1.3, 0.7))
    _check(_shape(dtype, 64, 9, 12, 0), beta=0.5)
    _check(_shape(dtype, 32, 9, 12, 0), beta=0.85)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("grid", [(1, 1), (1, 7), (9, 1), (57, 55), (4, 64), (5, 65), (3, 130)])
def test_grids(dtype, grid):
    """Ragged and narrow grids; rows of 64 tokens and wider (the window-row
    staging of the bf16 statistics pass holds grids up to 64 wide, wider ones
    read their window rows from global memory)."""
    _check(_shape(dtype, 64, grid[0], grid[1], 3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_structured_and_without_feature_map(dtype):
    _check(_shape(dtype, 64, 24, 20, 3, alpha="0.5"), structured=True)
    _check(_shape(dtype, 64, 11, 13, 3), relu=False)


@pytest.mark.parametrize("alpha", [0.0, 1.0])
def test_single_branch(alpha):
    _check(_shape("f32", 32, 10, 11, 3), alpha=alpha)


def test_full_size_pvt_layer():
    """The PVT stage-1 layer (32 slices, 56 x 56, d = 64, bf16, T = 3)."""
    shape = SHAPES["pvt_t_s1_56x56_T3"]
    _check(shape)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_walk_only_structured(dtype):
    """alpha = 1: dXq and dXk come from the walk alone.  Structured inputs,
    T = 3 and the deep walk T = 5, beta = 0.9; the untruncated walk."""
    _check(_shape(dtype, 64, 24, 20, 3, alpha="0.5"), structured=True, alpha=1.0)
    _check(_shape(dtype, 64, 24, 20, 5, alpha="0.5"), structured=True, alpha=1.0, beta=0.9)
    _check(_shape(dtype, 64, 24, 20, 0, alpha="0.5"), structured=True, alpha=1.0, beta=0.9)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [32, 64])
def test_walk_only_deep_small_grid(dtype, d):
    """alpha = 1 on i.i.d. inputs of a small grid with a deep walk."""
    _check(_shape(dtype, d, 9, 12, 5, alpha="0.5"), alpha=1.0, beta=0.9)
    _check(_shape(dtype, d, 7, 9, 3, alpha="0.5"), alpha=1.0)


def test_walk_only_full_size_pvt_layer():
    """alpha = 1 on the PVT stage-1 layer, i.i.d. and structured inputs."""
    _check(SHAPES["pvt_t_s1_56x56_T3"], alpha=1.0)
    _check(_shape("bf16", 64, 56, 56, 5, B=4, heads=1, alpha="0.5"), structured=True, alpha=1.0, beta=0.9)


def test_deterministic_and_empty():
    from hop_stochastic_vision_gb300 import lisa
    shape = _shape("bf16", 64, 28, 28, 3, B=4, heads=3)
    inp = to_device(make_inputs(shape))
    dO = _upstream(shape, 4, 3).cuda()
    a = lisa.backward(inp["xq"], inp["xk"], inp["v"], dO, (28, 28), 3, alpha=inp["alpha"], beta=0.5)
    b = lisa.backward(inp["xq"], inp["xk"], inp["v"], dO, (28, 28), 3, alpha=inp["alpha"], beta=0.5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q = torch.empty(0, 3, 196, 64, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv, da = lisa.backward(q, q, q, q, (14, 14), 3, alpha=torch.full((3,), 0.5, device="cuda"),
                                   beta=0.5)
    assert dq.shape == q.shape and torch.equal(da.cpu(), torch.zeros(3))


def test_captured_in_a_cuda_graph():
    """For bf16 at d = 64 the backward forks its dUbar launch onto a
    library-owned stream and joins it back into the caller's.  Captured in a
    CUDA graph (the fork and the join inside the capture) and replayed, it
    gives the eager call's bits; replayed on new inputs copied into the
    captured buffers, that input's eager bits."""
    from hop_stochastic_vision_gb300 import lisa
    shape = _shape("bf16", 64, 28, 28, 3, B=4, heads=3)
    sets = [(to_device(make_inputs(shape, seed=s)), _upstream(shape, 4, 3, seed=s + 1).cuda()) for s in (0, 1)]

    def run(inp, dO):
        return lisa.backward(inp["xq"], inp["xk"], inp["v"], dO, (28, 28), 3, alpha=inp["alpha"], beta=0.5)

    eager = [run(*x) for x in sets]   # the first eager call also creates the second stream
    torch.cuda.synchronize()
    inp = {k: v.clone() for k, v in sets[0][0].items()}
    dO = sets[0][1].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up on the capture stream
        run(inp, dO)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = run(inp, dO)
    for j, (x, y) in enumerate(sets):
        for key in ("xq", "xk", "v", "alpha"):
            inp[key].copy_(x[key])
        dO.copy_(y)
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip(outs, eager[j]):
            assert torch.equal(got, want), j


# -- adaptive (MLP) walk weights: lisa_backward_mlp ----------------------------------------

def _check_mlp(dtype, d, H, W, T, *, B=2, heads=2, hidden=32, scale=1.0, seed=0, relu=True, alpha=None,
               structured=False):
    from hop_stochastic_vision_gb300 import lisa
    shape = LayerShape("bwd_mlp", dtype, B, heads, H, W, d, T, "mlp", alpha="uniform(0.3,0.7)", hidden=hidden)
    inp = make_inputs(shape, seed=seed, structured=structured)
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], float(alpha))
    for key in ("W1", "b1", "W2", "b2"):   # the paper's N(0, 0.02) init, optionally scaled up
        inp[key] = inp[key] * scale
    if not relu:
        inp["xq"], inp["xk"] = inp["xq"].clamp_min(0), inp["xk"].clamp_min(0)
    dO = _upstream(shape, B, heads)
    dev = to_device(inp)
    mlp_dev = tuple(dev[k] for k in ("W1", "b1", "W2", "b2"))
    dq, dk, dv, da, pg = lisa.backward(dev["xq"], dev["xk"], dev["v"], dO.cuda(), (H, W), T, alpha=dev["alpha"],
                                       mlp=mlp_dev, relu=relu)
    torch.cuda.synchronize()
    mlp = tuple(inp[k].double().numpy() for k in ("W1", "b1", "W2", "b2"))
    want = oracle.backward(to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"]), to_f64(dO), (H, W), T,
                           alpha=inp["alpha"].double().numpy(), mlp=mlp, relu=relu)
    got = [to_f64(x.cpu()) for x in (dq, dk, dv)]
    for g in got:
        assert np.isfinite(g).all()
    err = max(assert_per_tensor(got, want[:3], shape))
    ptol = 1e-3 if dtype == "f32" else 2e-2
    for name, g, ref in zip(("dW1", "db1", "dW2", "db2"), pg, want[4]):
        g = g.cpu().double().numpy()
        scale_ref = max(np.abs(ref).max(), 1e-30)
        assert np.abs(g - ref).max() <= ptol * scale_ref, "%s err %.3e" % (name, np.abs(g - ref).max() / scale_ref)
    np.testing.assert_allclose(da.cpu().double().numpy(), want[3], rtol=1e-3, atol=1e-3 * np.abs(want[3]).max())
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
def test_mlp_widths(dtype, d):
    _check_mlp(dtype, d, 7, 9, 3, scale=20.0)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_mlp_depths(T):
    _check_mlp("f32", 32, 10, 11, T, scale=20.0)
    _check_mlp("bf16", 64, 10, 11, T, scale=20.0)


def test_mlp_hidden64_paper_init_and_no_feature_map():
    _check_mlp("bf16", 64, 9, 12, 4, hidden=64, scale=20.0)
    _check_mlp("bf16", 64, 12, 12, 3)                       # the paper's N(0, 0.02) init
    _check_mlp("f32", 32, 8, 9, 3, scale=20.0, relu=False)


def test_mlp_ragged_grid_and_full_size_deit384():
    _check_mlp("bf16", 64, 57, 55, 3, B=1, heads=2, scale=20.0)
    _check_mlp("bf16", 64, 24, 24, 3, B=64, heads=3, scale=20.0)   # the DeiT-T/384 layer's shape


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mlp_walk_only(dtype):
    """alpha = 1 with adaptive weights: the walk's and the MLP's gradients alone."""
    _check_mlp(dtype, 64, 24, 20, 5, scale=20.0, alpha=1.0, structured=True)
    _check_mlp(dtype, 64, 9, 12, 5, scale=20.0, alpha=1.0)
