"""GPU parity with the ELU(x) + 1 feature map (relu_inputs = 2): the forward
and the backward against the oracle's pinned ELU + 1 route.  The map is the
reading taken of the note's ELU feature map (section 2.1; paper Table 8); the
library serves it with its SIMT kernels for every dtype.  Tolerances as for
the ReLU layer."""
import numpy as np
import pytest
import torch

import oracle
from lisa_synth import LayerShape, make_inputs, to_f64

from helpers import TOL, max_rel_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa
    build.build()
    lisa.load()


def _shape(dtype, d, H, W, T, weights="geometric", B=2, heads=2):
    return LayerShape("elu", dtype, B, heads, H, W, d, T, weights, alpha="uniform(0.3,0.7)")


@pytest.mark.parametrize("dtype,d", [("f32", 16), ("f32", 64), ("bf16", 32), ("bf16", 64)])
@pytest.mark.parametrize("T,weights", [(3, "geometric"), (0, "geometric"), (3, "mlp")])
def test_forward_elu(dtype, d, T, weights):
    shape = _shape(dtype, d, 9, 11, T, weights)
    inp = make_inputs(shape)
    got = to_f64(run_gpu(to_device(inp), (9, 11), T, weights, relu="elu1"))
    want = run_oracle(inp, (9, 11), T, weights, relu="elu1")
    assert max_rel_err(got, want) <= TOL[dtype]


def test_forward_elu_full_size_pvt_layer():
    shape = LayerShape("elu_pvt", "bf16", 32, 1, 56, 56, 64, 3, "geometric")
    inp = make_inputs(shape)
    got = to_f64(run_gpu(to_device(inp), (56, 56), 3, "geometric", relu="elu1"))
    assert max_rel_err(got, run_oracle(inp, (56, 56), 3, "geometric", relu="elu1")) <= TOL["bf16"]


@pytest.mark.parametrize("dtype,d", [("f32", 32), ("bf16", 64)])
@pytest.mark.parametrize("T,weights", [(3, "geometric"), (0, "geometric"), (4, "mlp")])
@pytest.mark.parametrize("alpha", [None, 1.0])
def test_backward_elu(dtype, d, T, weights, alpha):
    """Each of dXq, dXk, dV against the oracle on its own norm; alpha = 1
    leaves the walk's gradient alone in dXq and dXk."""
    from hop_stochastic_vision_gb300 import lisa
    shape = _shape(dtype, d, 8, 10, T, weights)
    inp = make_inputs(shape)
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], alpha)
    if weights == "mlp":
        for key in ("W1", "b1", "W2", "b2"):
            inp[key] = inp[key] * 20.0
    g = torch.Generator("cpu").manual_seed(7)
    dO = torch.randn(inp["v"].shape, generator=g).to(inp["v"].dtype)
    dev = to_device(inp)
    kw = {"mlp": tuple(dev[k] for k in ("W1", "b1", "W2", "b2"))} if weights == "mlp" else {"beta": 0.5}
    res = lisa.backward(dev["xq"], dev["xk"], dev["v"], dO.cuda(), (8, 10), T, alpha=dev["alpha"], relu="elu1",
                        **kw)
    torch.cuda.synchronize()
    okw = {"mlp": tuple(inp[k].double().numpy() for k in ("W1", "b1", "W2", "b2"))} if weights == "mlp" \
        else {"beta": 0.5}
    want = oracle.backward(to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"]), to_f64(dO), (8, 10), T,
                           alpha=inp["alpha"].double().numpy(), relu="elu1", **okw)
    got = [to_f64(x.cpu()) for x in res[:3]]
    for name, g, w in zip(("dXq", "dXk", "dV"), got, want[:3]):
        err = max_rel_err(g, w)
        assert err <= TOL[dtype], "%s err %.3e (%s)" % (name, err, dtype)
    np.testing.assert_allclose(res[3].cpu().double().numpy(), want[3], rtol=1e-3,
                               atol=1e-3 * np.abs(want[3]).max())
    if weights == "mlp":
        ptol = 1e-3 if dtype == "f32" else 2e-2
        for gp, ref in zip(res[4], want[4]):
            assert np.abs(gp.cpu().double().numpy() - ref).max() <= ptol * np.abs(ref).max()
