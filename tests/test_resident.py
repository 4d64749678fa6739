"""GPU parity of the single-kernel tensor-core forward (lisa_forward_resident,
a test hook: one thread-block cluster per slice, K resident in shared
memory, the local branch parked in tensor memory) against the
double-precision oracle.

That kernel serves bf16 layers with d = 64 and walk weights shared by all
tokens on grids with an even number of rows and 8..64 columns in steps of 8
whose slice fits the cluster's shared memory; lisa_forward itself runs the
two-kernel chain on these layers.  Every case compares element by element
with the oracle (max over slices of ||gpu - oracle||_inf / ||oracle||_inf
<= 2e-2).  The cases cover cluster sizes 1 to 8 (uneven block-row splits,
several waves of clusters), walk depths 1 to 16 and the untruncated walk,
fixed weights with negative entries, isolated hops on structured inputs,
both single branches, zero query and key rows, inputs already
feature-mapped, bit-for-bit repeatability, and the layers the hook
rejects."""
import numpy as np
import pytest
import torch

from lisa_synth import SHAPES, LayerShape, make_inputs, to_f64

from helpers import TOL, max_rel_err, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa
    build.build()
    lisa.load()


def _run_resident(d, grid, T, *, beta=0.5, w=None, mlp=False, relu=True, eps=1e-6, expect=None):
    """lisa_forward_resident on device inputs; returns O (or the status when
    ``expect`` names the status the call must return)."""
    from hop_stochastic_vision_gb300 import lisa
    q, k, v = d["xq"], d["xk"], d["v"]
    B, heads, n, D = q.shape
    H, W = grid
    dt = lisa.LISA_BF16 if q.dtype == torch.bfloat16 else lisa.LISA_F32
    if mlp:
        wt, keep = lisa.make_weights(T, mlp=tuple(d[k] for k in ("W1", "b1", "W2", "b2")))
    elif w is not None:
        wt, keep = lisa.make_weights(T, w=list(w))
    else:
        wt, keep = lisa.make_weights(T, beta=beta)
    nbytes = lisa.lisa_workspace_bytes(B, heads, H, W, D, D, T, dt)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    out = torch.full_like(v, float("nan"))
    rc = lisa.lisa_forward_resident(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, heads, H,
                                    W, D, D, T, wt, d["alpha"].data_ptr(), eps, lisa.feature_map_code(relu),
                                    dt, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    del keep
    if expect is not None:
        assert rc == expect, lisa.lisa_status_string(rc)
        return rc
    assert rc == lisa.LISA_OK, lisa.lisa_status_string(rc)
    assert lisa.lisa_query_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == lisa.LISA_OK
    return out


def _check(shape, *, w=None, structured=False, alpha=None, relu=True, seed=0, zero=None):
    inp = make_inputs(shape, seed=seed, structured=structured)
    if alpha is not None:
        inp["alpha"] = torch.full_like(inp["alpha"], float(alpha))
    if not relu:
        inp["xq"], inp["xk"] = inp["xq"].clamp_min(0), inp["xk"].clamp_min(0)
    if zero is not None:
        inp[zero][:, :, ::3] = 0
    grid = (shape.H, shape.W)
    got = to_f64(_run_resident(to_device(inp), grid, shape.T, beta=shape.beta, w=w, relu=relu))
    want = run_oracle(inp, grid, shape.T, "geometric", beta=shape.beta, w=w, relu=relu)
    assert np.isfinite(got).all()
    err = max_rel_err(got, want)
    assert err <= TOL["bf16"], "max rel err %.3e (%s)" % (err, shape)
    return got, want


def _shape(B, heads, H, W, T=3, beta=0.5, alpha="uniform(0.3,0.7)"):
    return LayerShape("resident", "bf16", B, heads, H, W, 64, T, "geometric", beta=beta, alpha=alpha)


@pytest.mark.parametrize("T", [3, 5])
def test_pvt_layer_full_size(T):
    _check(SHAPES["pvt_t_s1_56x56_T%d" % T])


@pytest.mark.parametrize("B,heads,H,W", [(1, 1, 56, 56), (3, 1, 10, 16), (2, 1, 12, 8), (1, 1, 2, 8),
                                         (8, 1, 20, 24), (16, 1, 26, 40), (4, 1, 64, 48), (10, 4, 28, 32),
                                         (40, 1, 14, 8), (100, 2, 4, 56)])
def test_cluster_splits_and_grids(B, heads, H, W):
    """Cluster sizes 1..8, block-row splits that are not even, a second wave
    of clusters (200 slices) and the smallest grid (2 x 8)."""
    _check(_shape(B, heads, H, W))


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_depths(T):
    _check(_shape(4, 2, 16, 24, T=T, beta=0.7))


def test_fixed_weights_with_negative_entries():
    w = (0.2, -0.5, 1.3, 0.7)
    _check(_shape(4, 2, 18, 32, T=4), w=w)


@pytest.mark.parametrize("w", [(0.0, 1.0), (0.0, 0.0, 1.0), (0.0, 0.0, 0.0, 1.0)])
def test_isolated_hops_structured(w):
    """alpha = 1 and one-hot weights: the output is S^k V alone, on inputs
    whose transition is close to block-diagonal (the hops differ from mean V)."""
    _check(_shape(2, 2, 24, 24, T=len(w), alpha="0.5"), w=w, structured=True, alpha=1.0)


def test_structured_full_mix():
    _check(_shape(4, 1, 56, 56, T=5, beta=0.9, alpha="0.5"), structured=True)


@pytest.mark.parametrize("alpha", [0.0, 1.0])
def test_single_branch(alpha):
    _check(_shape(4, 2, 22, 48), alpha=alpha)


def test_T1_alpha1_returns_V_exactly():
    shape = _shape(4, 2, 20, 24, T=1)
    got, _ = _check(shape, alpha=1.0)
    inp = make_inputs(shape)
    assert np.array_equal(got, to_f64(inp["v"]))


@pytest.mark.parametrize("which", ["xq", "xk"])
def test_zero_query_and_key_rows(which):
    _check(_shape(4, 2, 16, 16), zero=which)


def test_prefeature_mapped_inputs():
    _check(_shape(4, 2, 16, 40), relu=False)


def test_deterministic():
    shape = SHAPES["pvt_t_s1_56x56_T3"]
    d = to_device(make_inputs(shape, B=8))
    a = _run_resident(d, (56, 56), 3)
    b = _run_resident(d, (56, 56), 3)
    assert torch.equal(a, b)


@pytest.mark.parametrize("beta", [0.5, 0.9])
def test_untruncated_walk(beta):
    """T = 0: the walk's d x d solve runs inside the kernel."""
    _check(_shape(4, 1, 56, 56, T=0, beta=beta))


def test_matches_lisa_forward_on_the_pvt_layer():
    from hop_stochastic_vision_gb300 import lisa
    shape = SHAPES["pvt_t_s1_56x56_T5"]
    d = to_device(make_inputs(shape, B=8))
    a = to_f64(_run_resident(d, (56, 56), 5, beta=shape.beta))
    b = to_f64(lisa.forward(d["xq"], d["xk"], d["v"], (56, 56), 5, alpha=d["alpha"], beta=shape.beta))
    assert max_rel_err(a, b) <= TOL["bf16"]


@pytest.mark.parametrize("case", ["odd_rows", "wide", "ragged_cols", "d32", "f32", "mlp", "elu"])
def test_rejects_layers_it_does_not_serve(case):
    from hop_stochastic_vision_gb300 import lisa
    H, W, D, dtype, weights, relu = 14, 16, 64, torch.bfloat16, "geometric", True
    if case == "odd_rows":
        H = 15
    elif case == "wide":
        W = 72
    elif case == "ragged_cols":
        W = 14
    elif case == "d32":
        D = 32
    elif case == "f32":
        dtype = torch.float32
    elif case == "elu":
        relu = "elu1"
    elif case == "mlp":
        weights = "mlp"
    shape = LayerShape("reject", "bf16", 2, 1, H, W, D, 3, weights, beta=0.5, alpha="0.5")
    inp = make_inputs(shape)
    d = to_device({k: (v.to(dtype) if k in ("xq", "xk", "v") else v) for k, v in inp.items()})
    _run_resident(d, (H, W), 3, mlp=weights == "mlp", relu=relu, expect=lisa.LISA_ERR_UNSUPPORTED)
