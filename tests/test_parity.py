"""GPU parity: liblisa.so against the double-precision oracle on the same
seeded inputs, element by element, at the layer shapes of the paper's
backbones (full size) and on small, ragged and degenerate cases.

Tolerance: max over slices of ||gpu - oracle||_inf / ||oracle||_inf,
1e-4 for fp32 layers and 2e-2 for bf16 layers (fp32 accumulation)."""
import numpy as np
import pytest
import torch

import oracle
from lisa_synth import SHAPES, LayerShape, make_inputs, to_f64

from helpers import TOL, max_rel_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa
    build.build()
    lisa.load()


def _check(shape: LayerShape, *, seed=0, B=None, heads=None, structured=False, w=None,
           relu=True, eps=1e-6, alpha=None, explicit=False, tol=None, mlp_scale=None):
    inp = make_inputs(shape, seed=seed, B=B, heads=heads, structured=structured)
    if mlp_scale is not None:
        for key in ("W1", "b1", "W2", "b2"):
            inp[key] = inp[key] * mlp_scale
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], float(alpha))
    if not relu:
        inp["xq"] = inp["xq"].clamp_min(0)
        inp["xk"] = inp["xk"].clamp_min(0)
    grid = (shape.H, shape.W)
    out = run_gpu(to_device(inp), grid, shape.T, shape.weights, beta=shape.beta, w=w, eps=eps,
                  relu=relu)
    got = to_f64(out)
    want = run_oracle(inp, grid, shape.T, shape.weights, beta=shape.beta, w=w, eps=eps, relu=relu)
    err = max_rel_err(got, want)
    limit = TOL[shape.dtype] if tol is None else tol
    assert np.isfinite(got).all()
    assert err <= limit, "max rel err %.3e > %.1e (%s)" % (err, limit, shape.name)
    if explicit:
        want_e = run_oracle(inp, grid, shape.T, shape.weights, beta=shape.beta, w=w, eps=eps,
                            relu=relu, mode=oracle.EXPLICIT)
        assert max_rel_err(got, want_e) <= limit
    return err


# -- the paper-shaped layers at full size ------------------------------------------

@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_shapes_full_size(name):
    shape = SHAPES[name]
    err = _check(shape, explicit=(shape.n <= 196 and shape.slices <= 4))
    print("full-size parity %s max_rel_err %.3e" % (name, err))


# -- small, ragged and odd grids -----------------------------------------------------

def _shape(dtype, d, H, W, T, weights="geometric", B=2, heads=2, alpha="uniform(0.3,0.7)", hidden=32):
    return LayerShape("case", dtype, B, heads, H, W, d, T, weights, alpha=alpha, hidden=hidden)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("grid", [(1, 1), (1, 7), (9, 1), (7, 9), (57, 55)])
def test_grids_and_widths(dtype, d, grid):
    _check(_shape(dtype, d, grid[0], grid[1], 3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 4, 5, 8])
def test_depths_geometric(dtype, T):
    _check(_shape(dtype, 32, 13, 11, T))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_adaptive_weights(dtype, d, T):
    _check(_shape(dtype, d, 10, 12, T, weights="mlp"), seed=T)


@pytest.mark.parametrize("hidden,T", [(32, 3), (32, 8), (64, 5), (20, 4)])
def test_adaptive_weights_far_from_uniform(hidden, T):
    """MLP parameters 25x the N(0, 0.02) init: hidden pre-activations of a
    few units and logits whose softmax is far from uniform, so the step
    weights (and the bf16 hi + lo split of W2 and h that forms the logits on
    the tensor path) matter to the output."""
    _check(_shape("bf16", 64, 14, 18, T, weights="mlp", hidden=hidden), seed=hidden + T, mlp_scale=25.0)


def test_limits_T16_and_hidden64():
    _check(_shape("f32", 16, 9, 9, 16))
    _check(_shape("bf16", 64, 9, 9, 8, weights="mlp", hidden=64))


def test_long_ragged_chunks():
    # n not a multiple of any tile size; several split-K chunks per slice
    _check(_shape("bf16", 64, 61, 67, 3, B=1, heads=3))
    _check(_shape("f32", 64, 61, 67, 5, B=1, heads=1))


# -- structured inputs and isolated hop terms -------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("w", [(0.0, 1.0), (0.0, 0.0, 1.0), (0.0, 0.0, 0.0, 1.0), (0.2, -0.5, 1.3)])
def test_isolated_hops_structured(dtype, w):
    """Fixed weights pick single S^k V terms on data whose transition matrix
    is close to block-diagonal, so the hop terms are far from mean(V)."""
    shape = _shape(dtype, 64 if dtype == "bf16" else 32, 24, 20, len(w), alpha="0.5")
    _check(shape, structured=True, w=w, alpha=1.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_structured_full_mix(dtype):
    _check(_shape(dtype, 64, 28, 28, 5, alpha="0.5"), structured=True)
    _check(_shape(dtype, 64, 28, 28, 3, weights="mlp", alpha="0.5"), structured=True)


# -- degenerate and special cases ---------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_T1_alpha1_returns_V_exactly(dtype):
    shape = _shape(dtype, 64, 14, 14, 1, alpha="0.5")
    inp = make_inputs(shape)
    inp["alpha"] = torch.ones_like(inp["alpha"])
    out = run_gpu(to_device(inp), (14, 14), 1, "geometric")
    assert torch.equal(out.cpu(), inp["v"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("alpha", [0.0, 1.0])
def test_single_branch(dtype, alpha):
    _check(_shape(dtype, 64, 15, 17, 3), alpha=alpha)
    _check(_shape(dtype, 64, 15, 17, 3, weights="mlp"), alpha=alpha)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constant_V(dtype):
    shape = _shape(dtype, 64, 12, 16, 5)
    inp = make_inputs(shape)
    inp["v"] = torch.full_like(inp["v"], 1.5)
    out = run_gpu(to_device(inp), (12, 16), 5, "geometric")
    assert torch.allclose(out.cpu().double(), torch.full(out.shape, 1.5, dtype=torch.float64),
                          rtol=TOL[dtype], atol=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_queries_and_zero_keys(dtype):
    shape = _shape(dtype, 32, 8, 9, 3)
    inp = make_inputs(shape)
    grid = (8, 9)
    for key in ("xq", "xk"):
        case = dict(inp)
        case[key] = -case[key].abs() - 0.5        # ReLU -> all zero
        got = to_f64(run_gpu(to_device(case), grid, 3, "geometric"))
        want = run_oracle(case, grid, 3, "geometric")
        assert max_rel_err(got, want) <= TOL[dtype], key
    # a single zero query row among live ones
    case = dict(inp)
    case["xq"] = case["xq"].clone()
    case["xq"][:, :, 5] = -1.0
    got = to_f64(run_gpu(to_device(case), grid, 3, "geometric"))
    assert max_rel_err(got, run_oracle(case, grid, 3, "geometric")) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefeature_mapped_inputs(dtype):
    _check(_shape(dtype, 64, 11, 13, 3), relu=False)


def test_eps_variants():
    _check(_shape("f32", 32, 9, 10, 3), eps=1e-2)
    _check(_shape("bf16", 64, 9, 10, 3), eps=1e-3)


def test_deterministic():
    shape = SHAPES["pvt_t_s1_56x56_T5"]
    d = to_device(make_inputs(shape, B=4))
    a = run_gpu(d, (56, 56), 5, "geometric")
    b = run_gpu(d, (56, 56), 5, "geometric")
    assert torch.equal(a, b)
    shape = SHAPES["deit_t384_24x24_mlp"]
    d = to_device(make_inputs(shape, B=4))
    assert torch.equal(run_gpu(d, (24, 24), 3, "mlp"), run_gpu(d, (24, 24), 3, "mlp"))


def test_empty_batch():
    from hop_stochastic_vision_gb300 import lisa
    q = torch.empty(0, 3, 196, 64, dtype=torch.bfloat16, device="cuda")
    out = lisa.forward(q, q, q, (14, 14), 3, alpha=torch.full((3,), 0.5, device="cuda"), beta=0.5)
    assert out.shape == q.shape


def test_forward_host_matches_device_path():
    from hop_stochastic_vision_gb300 import lisa
    shape = SHAPES["deit_t_14x14"]
    inp = make_inputs(shape, B=8)
    d = to_device(inp)
    ref = run_gpu(d, (14, 14), 3, "geometric")
    hq, hk, hv = (inp[k].pin_memory() for k in ("xq", "xk", "v"))
    ho = torch.empty_like(hv).pin_memory()
    dq, dk, dv, do = (torch.empty_like(d["v"]) for _ in range(4))
    B, heads, n, D = hq.shape
    wt, keep = lisa.make_weights(3, beta=0.5)
    nb = lisa.lisa_workspace_bytes(B, heads, 14, 14, D, D, 3, lisa.LISA_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = lisa.lisa_forward_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(),
                                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), B, heads,
                                14, 14, D, D, 3, wt, d["alpha"].data_ptr(), 1e-6, 1, lisa.LISA_BF16,
                                ws.data_ptr(), nb, st)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(ho, ref.cpu())
