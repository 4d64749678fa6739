"""GPU parity of the untruncated geometric walk (T = 0 at the C ABI):
g = (1-beta) (I - beta S)^-1 V, which the library evaluates through the d x d
system (I - beta M) X = U_1 of the push-through identity, against the
double-precision oracle's own solve, on every kernel chain that serves it
(SIMT fp32/bf16 for d = 16, 32, 64; the tensor-core chain with fused and
with split statistics for bf16 d = 64).

Tolerance as for the truncated layer: max over slices of
||gpu - oracle||_inf / ||oracle||_inf <= 1e-4 (fp32), 2e-2 (bf16)."""
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


def _shape(dtype, d, H, W, B=2, heads=2, alpha="uniform(0.3,0.7)"):
    return LayerShape("untruncated", dtype, B, heads, H, W, d, 0, "geometric", alpha=alpha)


def _check(shape, *, beta=0.5, seed=0, structured=False, alpha=None, explicit=False):
    inp = make_inputs(shape, seed=seed, structured=structured)
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], float(alpha))
    grid = (shape.H, shape.W)
    got = to_f64(run_gpu(to_device(inp), grid, 0, "geometric", beta=beta))
    want = run_oracle(inp, grid, 0, "geometric", beta=beta)
    err = max_rel_err(got, want)
    assert np.isfinite(got).all()
    assert err <= TOL[shape.dtype], "max rel err %.3e (beta %g, %s)" % (err, beta, shape.dtype)
    if explicit:
        want_e = run_oracle(inp, grid, 0, "geometric", beta=beta, mode=oracle.EXPLICIT)
        assert max_rel_err(got, want_e) <= TOL[shape.dtype]
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("beta", [0.0, 0.5, 0.9])
def test_widths_and_beta(dtype, d, beta):
    _check(_shape(dtype, d, 11, 13), beta=beta, explicit=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("grid", [(1, 1), (1, 9), (7, 1), (57, 55)])
def test_grids(dtype, grid):
    _check(_shape(dtype, 64, grid[0], grid[1]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("beta", [0.5, 0.95])
def test_structured_global_only(dtype, beta):
    """Near block-diagonal S, alpha = 1: the hop terms carry the output."""
    _check(_shape(dtype, 64, 24, 20, alpha="0.5"), beta=beta, structured=True, alpha=1.0)


def test_full_size_pvt_fused_statistics():
    """The PVT stage-1 layer (32 slices, 56 x 56, d = 64, bf16): fused statistics."""
    shape = SHAPES["pvt_t_s1_56x56_T3"]
    _check(LayerShape("pvt_untruncated", "bf16", shape.B, shape.heads, 56, 56, 64, 0, "geometric"))


def test_long_slices_split_statistics():
    """Few slices of 128 x 128 tokens: more chunks than a cluster holds, so the
    statistics run split-K and the solve sits in the separate recurrence kernel."""
    _check(LayerShape("long_untruncated", "bf16", 1, 4, 128, 128, 64, 0, "geometric"), beta=0.8)
    _check(LayerShape("long_untruncated", "f32", 1, 2, 96, 96, 32, 0, "geometric"), beta=0.8)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_beta0_alpha1_returns_V_exactly(dtype):
    shape = _shape(dtype, 64, 14, 14)
    inp = make_inputs(shape)
    inp["alpha"] = torch.ones_like(inp["alpha"])
    out = run_gpu(to_device(inp), (14, 14), 0, "geometric", beta=0.0)
    assert torch.equal(out.cpu(), inp["v"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constant_V(dtype):
    shape = _shape(dtype, 64, 12, 16)
    inp = make_inputs(shape)
    inp["v"] = torch.full_like(inp["v"], -0.75)
    out = run_gpu(to_device(inp), (12, 16), 0, "geometric", beta=0.7)
    assert torch.allclose(out.cpu().double(), torch.full(out.shape, -0.75, dtype=torch.float64),
                          rtol=TOL[dtype], atol=0)


def test_approaches_long_truncated_walk():
    """On the GPU too, the untruncated layer is the limit of the truncated one:
    T = 16 at beta = 0.5 differs from it by ~beta^16 of the hop terms."""
    shape = _shape("f32", 32, 13, 11)
    d = to_device(make_inputs(shape))
    a = to_f64(run_gpu(d, (13, 11), 0, "geometric", beta=0.5))
    b = to_f64(run_gpu(d, (13, 11), 16, "geometric", beta=0.5))
    assert max_rel_err(a, b) <= 1e-4
